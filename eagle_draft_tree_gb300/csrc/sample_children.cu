// sample_children.cu -- the sampled children of draft rows (non-greedy drafting), sm_103a.
//
// Page: "EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty" (papercache.org),
// appendix A.1: in the non-greedy setting the k children of a node are sampled from the draft
// distribution rather than taken as its top k.  Children of a row x are k independent draws from
// q = softmax(x / T) with replacement, draw j by inverse CDF over ascending token id with the
// caller's uniform u_j, kept in draw order; a child's log-confidence is x_t / T - logsumexp(x / T),
// as for top-k children.  Children drawn this way are what makes build -> verify exactly lossless:
// multi-round speculative sampling tests candidates drawn from q.
//
// One thread-block cluster per row; its CTAs split the row into contiguous slices.
//   pass 1 (HBM)  slice maximum; the cluster reads its CTAs' maxima through distributed shared
//                 memory, so every CTA holds the row maximum M.
//   pass 2 (L2)   weights w = 2^((x - M) c) with c = log2(e) / T, each as an integer in units of
//                 2^-S (S = 62 - ceil(log2 V), so the row total stays below 2^62) and summed per
//                 4-token chunk, per (chunk column, warp) in shared memory and per slice for the
//                 cluster.  Integer sums are exact, so the slices' totals, their prefix sums and
//                 every CTA's view of the row total agree.
//   draw j        warp j of each CTA: target = floor(u_j * total) in fixed point; the CTA whose
//                 slice range holds it walks column -> warp -> lane -> token, re-deriving the one
//                 chunk's weights from the row with the same arithmetic (hence the same values).
// A weight's exponent is formed without rounding error: x - M by an error-free sum (Knuth's
// TwoSum) and its product with c = c_hi + c_lo by an error-free FMA product, split into an integer
// n and a fraction f in [-1/2, 1/2] rounded once; w = 2^n 2^f with 2^f from the SFU (ex2.approx,
// whose relative error on [-1/2, 1/2] eagle_selftest_exp2_error measures).  A step of the row's
// CDF is then off by at most half the weights' relative error plus V 2^-S.
// The row's log normaliser is M / T + ln(total 2^-S).  Chunks start at multiples of 4 tokens and
// every sum above a weight is exact, so draws and log-confidences do not depend on the slicing.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace eagle {

int splits_for_rows(long rows, int vocab);

namespace {

constexpr int kSmpThreads = 512;
constexpr int kSmpWarps = kSmpThreads / 32;
constexpr int kSmpMaxCols = 128;                           // chunk columns per slice
constexpr int kSmpMaxSlice = kSmpMaxCols * kSmpThreads * 4;  // 262144 tokens
constexpr int kSmpMaxSplits = 8;
constexpr double kLn2 = 0.69314718055994530942;

// Warp-wide exact sum of 64-bit values whose total is below 2^64 (the result in every lane):
// three 32-bit reductions of 22-bit parts.
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
    const uint32_t p0 = __reduce_add_sync(0xffffffffu, uint32_t(v) & 0x3fffffu);
    const uint32_t p1 = __reduce_add_sync(0xffffffffu, uint32_t(v >> 22) & 0x3fffffu);
    const uint32_t p2 = __reduce_add_sync(0xffffffffu, uint32_t(v >> 44));
    return (uint64_t(p2) << 44) + (uint64_t(p1) << 22) + p0;
}

// Two floats in one 64-bit register pair, for the paired f32x2 arithmetic of sm_100-class SMs
// (each operation rounds each lane exactly as its scalar form would).
__device__ __forceinline__ uint64_t x2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void x2_split(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t x2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t x2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// b - a, rounded once (a times -1 is exact)
__device__ __forceinline__ uint64_t x2_sub(uint64_t b, uint64_t a) { return x2_fma(a, x2(-1.f, -1.f), b); }

// floor(p 2^e) for a normal p (the SFU's 2^f, in [0.70, 1.42]) and e <= S, exactly, on the
// integer pipe: p = m 2^(ex - 150) with a 24-bit m, so p 2^e = m 2^(ex - 150 + e).
__device__ __forceinline__ uint64_t scaled_floor(float p, int e) {
    const uint32_t bits = __float_as_uint(p);
    const uint32_t m = (bits & 0x7fffffu) | 0x800000u;
    const int sh = int(bits >> 23) - 150 + e;
    return sh >= 0 ? (uint64_t(m) << sh) : (sh > -24 ? uint64_t(m >> (-sh)) : 0ull);
}

// The fixed-point weights floor(2^((x - M) c) 2^S) of two logits x <= M (0 for -inf or past
// 2^-S): x - M by TwoSum, times c = c_hi + c_lo by an FMA product, r = n + f with n = rint(r_hi)
// and f rounded once; 2^f in [0.70, 1.42] from the SFU (its only instruction there), then
// 2^(n + S) applied exactly.
__device__ __forceinline__ void weight_fx2(float xa, float xb, float M, float c_hi, float c_lo, int S, uint64_t &wa,
                                           uint64_t &wb) {
    const uint64_t X = x2(xa, xb), Mn = x2(-M, -M), C = x2(c_hi, c_hi);
    const uint64_t D = x2_add(X, Mn);  // TwoSum(x, -M): D + E = x - M exactly
    const uint64_t BB = x2_sub(D, X);
    const uint64_t E = x2_add(x2_sub(X, x2_sub(D, BB)), x2_sub(Mn, BB));
    const uint64_t RH = x2_mul(D, C);  // RH + RL = (D + E)(c_hi + c_lo) to ~2^-48
    const uint64_t RL = x2_add(x2_fma(D, C, x2_mul(RH, x2(-1.f, -1.f))),  // the product's rounding error
                               x2_fma(D, x2(c_lo, c_lo), x2_mul(E, C)));
    // n = rint(RH) by adding 1.5 2^23 (whose ulp is 1) on the FMA pipe; the sum's bits give n as
    // an integer (|RH| < 2^22 wherever the weight is kept)
    const float kMagic = 12582912.0f;
    const uint64_t TN = x2_add(RH, x2(kMagic, kMagic));
    const uint64_t N = x2_sub(TN, x2(kMagic, kMagic));
    float rha, rhb, ta, tb;
    x2_split(RH, rha, rhb);
    x2_split(TN, ta, tb);
    const int na = __float_as_int(ta) - __float_as_int(kMagic), nb = __float_as_int(tb) - __float_as_int(kMagic);
    float fa, fb;
    x2_split(x2_add(x2_sub(RH, N), RL), fa, fb);  // RH - n is exact
    float da, db;
    x2_split(D, da, db);
    // an infinite logit has no weight (its difference is NaN); one more than S + 2 octaves below
    // the maximum adds less than 2^-S
    wa = (xa == -INFINITY || !(da <= 0.f) || rha < -float(S + 2)) ? 0ull : scaled_floor(fast_exp2(fa), S + na);
    wb = (xb == -INFINITY || !(db <= 0.f) || rhb < -float(S + 2)) ? 0ull : scaled_floor(fast_exp2(fb), S + nb);
}

struct SampleArgs {
    const float *x;        // [B][R][V] rows
    const float *u;        // [B][R][k] uniforms
    int32_t *row_tok;      // [B][out_R][k]
    double *row_lc;        // [B][out_R][k]
    int32_t *status;
    int V, R, k, chunk, out_R, out_r0;
    int S;               // weights in units of 2^-S
    float c, c_lo;       // log2(e) / T as a float pair
    double inv_t;        // 1 / T
};

// Chunk q of a slice: the four values at lo + 4q .. lo + 4q + 3 (-inf past hi).
__device__ __forceinline__ float4 load_chunk(const float *row, int lo, int hi, int q, bool vec) {
    const int t = lo + 4 * q;
    if (vec) return __ldg(reinterpret_cast<const float4 *>(row + t));
    float4 v;
    v.x = t < hi ? __ldg(row + t) : -INFINITY;
    v.y = t + 1 < hi ? __ldg(row + t + 1) : -INFINITY;
    v.z = t + 2 < hi ? __ldg(row + t + 2) : -INFINITY;
    v.w = t + 3 < hi ? __ldg(row + t + 3) : -INFINITY;
    return v;
}

// The chunk's fixed-point weights against the row maximum and their total; the pass and the draw
// both call this, so they derive identical values.
__device__ __forceinline__ uint64_t chunk_w(float4 x, float M, const SampleArgs &a, uint64_t (&w)[4]) {
    weight_fx2(x.x, x.y, M, a.c, a.c_lo, a.S, w[0], w[1]);
    weight_fx2(x.z, x.w, M, a.c, a.c_lo, a.S, w[2], w[3]);
    return (w[0] + w[1]) + (w[2] + w[3]);
}

// Inclusive warp scan of 64-bit values.
__device__ __forceinline__ uint64_t warp_incl_scan(uint64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    return v;
}

// The lane whose step [incl - v, incl) holds `target` (relative to `base`); if none (cannot
// happen with exact sums) the last lane with a non-zero value.  -1 when no lane has weight.
__device__ __forceinline__ int claim_lane(uint64_t v, uint64_t incl, uint64_t base, uint64_t target, bool valid) {
    const unsigned hit = __ballot_sync(0xffffffffu, valid && v > 0 && base + incl - v <= target && target < base + incl);
    if (hit) return __ffs(hit) - 1;
    const unsigned nz = __ballot_sync(0xffffffffu, valid && v > 0);
    return nz ? 31 - __clz(nz) : -1;
}

__global__ void __launch_bounds__(kSmpThreads) row_sample_kernel(SampleArgs a) {
    pdl_wait();
    pdl_launch_next();
    __shared__ uint64_t s_col[kSmpMaxCols][kSmpWarps];  // per (column, warp) fixed-point totals
    __shared__ float s_wmax[kSmpWarps];
    __shared__ float s_max;     // this slice's maximum (read by the peers)
    __shared__ uint64_t s_tot;  // this slice's total (read by the peers)

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int splits = int(cluster.num_blocks());
    const int r = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *row = a.x + (size_t(b) * a.R + r) * size_t(a.V);
    const int lo = rank * a.chunk;
    const int hi = min(a.V, lo + a.chunk);
    const int cnt = hi > lo ? hi - lo : 0;
    const int nch = (cnt + 3) >> 2;
    const int ncol = (nch + kSmpThreads - 1) / kSmpThreads;
    const bool vec = ((a.V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0);

    // pass 1: the slice maximum
    float m = -INFINITY;
#pragma unroll 4
    for (int q = tid; q < nch; q += kSmpThreads) {
        const float4 v = load_chunk(row, lo, hi, q, vec);
        m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) s_wmax[warp] = m;
    __syncthreads();
    if (tid == 0) {
        float mm = -INFINITY;
        for (int w = 0; w < kSmpWarps; ++w) mm = fmaxf(mm, s_wmax[w]);
        s_max = mm;
    }
    cluster.sync();
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, *cluster.map_shared_rank(&s_max, s));

    // pass 2: fixed-point totals per (column, warp), then the slice total
    // (four columns' loads in flight at a time; the trip counts are CTA-uniform, so every lane
    // reaches the warp sums)
    for (int e0 = 0; e0 < ncol; e0 += 4) {
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int q = tid + (e0 + i) * kSmpThreads;
            v[i] = (e0 + i < ncol && q < nch) ? load_chunk(row, lo, hi, q, vec)
                                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (e0 + i >= ncol) break;
            uint64_t w[4];
            const uint64_t t = warp_sum_u64(M == -INFINITY ? 0ull : chunk_w(v[i], M, a, w));
            if (lane == 0) s_col[e0 + i][warp] = t;
        }
    }
    __syncthreads();
    if (warp == 0) {
        uint64_t t = 0;
        for (int i = lane; i < ncol * kSmpWarps; i += 32) t += s_col[i / kSmpWarps][i % kSmpWarps];
        t = warp_sum_u64(t);
        if (lane == 0) s_tot = t;
    }
    cluster.sync();
    uint64_t total = 0, excl = 0;
    for (int s = 0; s < splits; ++s) {
        const uint64_t t = *cluster.map_shared_rank(&s_tot, s);
        if (s < rank) excl += t;
        total += t;
    }
    // the peers may leave once every CTA has read the totals: the draws read only this CTA's own
    // shared memory and global memory
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    const uint64_t mine = s_tot;

    // draws: warp j takes draw j
    if (warp < a.k) {
        const int j = warp;
        const size_t urow = (size_t(b) * a.R + r) * a.k;
        float u = __ldg(a.u + urow + j);
        u = u > 0.f ? fminf(u, 0.99999994f) : 0.f;  // [0, 1); NaN -> 0
        const size_t o = (size_t(b) * a.out_R + a.out_r0 + r) * a.k + j;
        if (total == 0) {  // no finite logit in the row
            if (rank == 0 && lane == 0) {
                a.row_tok[o] = 0;
                a.row_lc[o] = -INFINITY;
                set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
            }
        } else {
            const uint64_t target = scale_fx(total, u);  // < total
            if (excl <= target && target < excl + mine) {
                const uint64_t local = target - excl;
                // column (warp-uniform loop: `hit` is a ballot)
                uint64_t base = 0;
                int col = 0;
                for (int e0 = 0; e0 < ncol; e0 += 32) {
                    const int e = e0 + lane;
                    uint64_t v = 0;
                    if (e < ncol)
#pragma unroll
                        for (int w = 0; w < kSmpWarps; ++w) v += s_col[e][w];
                    const uint64_t incl = warp_incl_scan(v);
                    const unsigned hit =
                        __ballot_sync(0xffffffffu, v > 0 && base + incl - v <= local && local < base + incl);
                    if (hit) {
                        const int l = __ffs(hit) - 1;
                        col = e0 + l;
                        base += __shfl_sync(0xffffffffu, incl - v, l);
                        break;
                    }
                    base += __shfl_sync(0xffffffffu, incl, 31);
                }
                // warp within the column
                {
                    const uint64_t v = lane < kSmpWarps ? s_col[col][lane] : 0ull;
                    const uint64_t incl = warp_incl_scan(v);
                    int l = claim_lane(v, incl, base, local, lane < kSmpWarps);
                    if (l < 0) l = 0;
                    base += __shfl_sync(0xffffffffu, incl - v, l);
                    // lane within the warp: chunk q of the slice
                    const int q = col * kSmpThreads + l * 32 + lane;
                    uint64_t w[4] = {0ull, 0ull, 0ull, 0ull};
                    const uint64_t cv = q < nch ? chunk_w(load_chunk(row, lo, hi, q, vec), M, a, w) : 0ull;
                    const uint64_t cincl = warp_incl_scan(cv);
                    int cl = claim_lane(cv, cincl, base, local, q < nch);
                    if (cl < 0) cl = 0;
                    if (lane == cl) {
                        // inside the chunk: the exact prefix sums of its fixed-point weights
                        const uint64_t rem = local >= base + cincl - cv ? local - (base + cincl - cv) : 0ull;
                        const uint64_t a1 = w[0] + w[1], a2 = a1 + w[2], a3 = a2 + w[3];
                        int lastp = 0;
                        if (w[1] > 0) lastp = 1;
                        if (w[2] > 0) lastp = 2;
                        if (w[3] > 0) lastp = 3;
                        const int i = (w[0] > 0 && w[0] > rem)   ? 0
                                      : (w[1] > 0 && a1 > rem) ? 1
                                      : (w[2] > 0 && a2 > rem) ? 2
                                      : (w[3] > 0 && a3 > rem) ? 3
                                                               : lastp;
                        const int tok = min(lo + 4 * q + i, hi - 1);  // in range even on a fallback
                        const double lse = double(M) * a.inv_t + (ln_pos(double(total)) - a.S * kLn2);
                        a.row_tok[o] = tok;
                        a.row_lc[o] = double(__ldg(row + tok)) * a.inv_t - lse;
                    }
                }
            }
        }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Self-test of the SFU exponential the draws use: the largest relative error of ex2.approx over
// every float f with |f| <= 1/2 (the fractions weight_fx passes it), against the double-precision
// exp2, as the bits of a non-negative float (atomicMax on them orders like the floats).
__global__ void __launch_bounds__(256) exp2_error_kernel(uint32_t *out) {
    float worst = 0.f;
    const uint32_t top = 0x3f000000u;  // 0.5
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i <= 2ull * top + 1;
         i += uint64_t(gridDim.x) * blockDim.x) {
        const uint32_t mag = uint32_t(i >> 1);
        const float f = __uint_as_float(mag | ((i & 1) ? 0x80000000u : 0u));
        const double ref = exp2(double(f));
        const double got = double(fast_exp2(f));
        worst = fmaxf(worst, float(fabs(got - ref) / ref));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, off));
    if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(worst));
}

}  // namespace

eagle_status exp2_error_launch(float *out, cudaStream_t stream) {
    if (cudaMemsetAsync(out, 0, sizeof(float), stream) != cudaSuccess) return EAGLE_ERR_CUDA;
    exp2_error_kernel<<<device_sm_count() * 8, 256, 0, stream>>>(reinterpret_cast<uint32_t *>(out));
    if (cudaPeekAtLastError() != cudaSuccess) return EAGLE_ERR_CUDA;
    note_launch();
    return EAGLE_OK;
}

size_t row_sample_max_vocab() { return size_t(kSmpMaxSlice) * kSmpMaxSplits; }

// The k sampled children of R rows of B sequences (uniforms u [B][R][k]) into
// row_tok / row_lc [B][out_R][k] at rows out_r0 .. out_r0 + R - 1.
eagle_status row_sample_launch(const float *draft, const float *u, int B, int R, int V, int k, float tree_temp,
                               int32_t *row_tok, double *row_lc, int out_R, int out_r0, int32_t *status,
                               cudaStream_t stream) {
    if (size_t(V) > row_sample_max_vocab() || k > kSmpWarps) return EAGLE_ERR_UNSUPPORTED;
    int splits = splits_for_rows(long(B) * R, V);
    const int need = (V + kSmpMaxSlice - 1) / kSmpMaxSlice;
    if (splits < need) splits = need;
    if (splits > kSmpMaxSplits) splits = kSmpMaxSplits;
    int chunk = (V + splits - 1) / splits;
    chunk = (chunk + 3) & ~3;
    SampleArgs sa;
    sa.x = draft;
    sa.u = u;
    sa.row_tok = row_tok;
    sa.row_lc = row_lc;
    sa.status = status;
    sa.V = V;
    sa.R = R;
    sa.k = k;
    sa.chunk = chunk;
    sa.out_R = out_R;
    sa.out_r0 = out_r0;
    const double cd = 1.4426950408889634074 / double(tree_temp);
    sa.c = float(cd);
    sa.c_lo = float(cd - double(sa.c));
    int lv = 0;  // ceil(log2 V)
    while ((1l << lv) < long(V)) ++lv;
    sa.S = 62 - lv;
    sa.inv_t = 1.0 / double(tree_temp);
    if (launch_pdl(row_sample_kernel, dim3(splits, R, B), dim3(kSmpThreads), 0, stream, unsigned(splits), sa) !=
        cudaSuccess)
        return EAGLE_ERR_CUDA;
    note_launch();
    return EAGLE_OK;
}

}  // namespace eagle
