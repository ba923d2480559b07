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
//   pass 2 (L2)   weights w = 2^((x - M) c) with c = log2(e) / T, summed per 4-token chunk in float
//                 and then as integers in units of 2^-40: per (chunk column, warp) totals stay in
//                 shared memory, slice totals go to the cluster.  Integer sums are exact, so the
//                 slices' totals, their prefix sums and every CTA's view of the row total agree.
//   draw j        warp j of each CTA: target = floor(u_j * total) in fixed point; the CTA whose
//                 slice range holds it walks column -> warp -> lane -> token, re-deriving the one
//                 chunk's weights from the row with the same arithmetic (hence the same values).
// The row's log normaliser is M / T + ln(total 2^-40).  Chunks start at multiples of 4 tokens and
// every sum above a chunk is exact, so draws and log-confidences do not depend on the slicing.
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
constexpr float kFx40 = 1099511627776.0f;  // 2^40
constexpr double kLn2_40 = 40.0 * 0.69314718055994530942;

// floor(x 2^40) for x in [0, 4] (NaN and non-positive give 0; larger values are clamped).
__device__ __forceinline__ uint64_t fx40(float x) {
    if (!(x > 0.f)) return 0ull;
    const uint32_t bits = __float_as_uint(fminf(x, 4.f));
    const int ex = int(bits >> 23);  // x = m 2^(ex - 150), so x 2^40 = m 2^(ex - 110)
    const uint32_t m = (bits & 0x7fffffu) | 0x800000u;
    return ex >= 110 ? (uint64_t(m) << (ex - 110)) : (ex > 86 ? uint64_t(m >> (110 - ex)) : 0ull);
}

struct SampleArgs {
    const float *x;        // [B][R][V] rows
    const float *u;        // [B][R][k] uniforms
    int32_t *row_tok;      // [B][out_R][k]
    double *row_lc;        // [B][out_R][k]
    int32_t *status;
    int V, R, k, chunk, out_R, out_r0;
    float c;       // log2(e) / T
    double inv_t;  // 1 / T
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

// The chunk's weights against the row maximum (0 for -inf) and its fixed-point total; the pass
// and the draw both call this, so they derive identical values.
__device__ __forceinline__ uint64_t chunk_w(float4 x, float c, float mc, float (&w)[4]) {
    w[0] = x.x == -INFINITY ? 0.f : fast_exp2(fmaf(x.x, c, -mc));
    w[1] = x.y == -INFINITY ? 0.f : fast_exp2(fmaf(x.y, c, -mc));
    w[2] = x.z == -INFINITY ? 0.f : fast_exp2(fmaf(x.z, c, -mc));
    w[3] = x.w == -INFINITY ? 0.f : fast_exp2(fmaf(x.w, c, -mc));
    return fx40(((w[0] + w[1]) + w[2]) + w[3]);
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
    const float c = a.c;

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
    const float mc = M == -INFINITY ? 0.f : M * c;

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
            float w[4];
            const uint64_t t = warp_sum_fx(chunk_w(v[i], c, mc, w));
            if (lane == 0) s_col[e0 + i][warp] = t;
        }
    }
    __syncthreads();
    if (warp == 0) {
        uint64_t t = 0;
        for (int i = lane; i < ncol * kSmpWarps; i += 32) t += s_col[i / kSmpWarps][i % kSmpWarps];
        t = warp_sum_fx(t);
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
                    float w[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint64_t cv = q < nch ? chunk_w(load_chunk(row, lo, hi, q, vec), c, mc, w) : 0ull;
                    const uint64_t cincl = warp_incl_scan(cv);
                    int cl = claim_lane(cv, cincl, base, local, q < nch);
                    if (cl < 0) cl = 0;
                    if (lane == cl) {
                        // inside the chunk: the float partial sums its total was formed from
                        const uint64_t rem = local >= base + cincl - cv ? local - (base + cincl - cv) : 0ull;
                        const float rr = float(rem) * (1.f / kFx40);
                        const float a1 = w[0] + w[1], a2 = a1 + w[2], a3 = a2 + w[3];
                        int lastp = 0;
                        if (w[1] > 0.f) lastp = 1;
                        if (w[2] > 0.f) lastp = 2;
                        if (w[3] > 0.f) lastp = 3;
                        const int i = (w[0] > 0.f && w[0] > rr)   ? 0
                                      : (w[1] > 0.f && a1 > rr) ? 1
                                      : (w[2] > 0.f && a2 > rr) ? 2
                                      : (w[3] > 0.f && a3 > rr) ? 3
                                                                : lastp;
                        const int tok = min(lo + 4 * q + i, hi - 1);  // in range even on a fallback
                        const double lse = double(M) * a.inv_t + (ln_pos(double(total)) - kLn2_40);
                        a.row_tok[o] = tok;
                        a.row_lc[o] = double(__ldg(row + tok)) * a.inv_t - lse;
                    }
                }
            }
        }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace

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
    sa.c = kLog2e / tree_temp;
    sa.inv_t = 1.0 / double(tree_temp);
    if (launch_pdl(row_sample_kernel, dim3(splits, R, B), dim3(kSmpThreads), 0, stream, unsigned(splits), sa) !=
        cudaSuccess)
        return EAGLE_ERR_CUDA;
    note_launch();
    return EAGLE_OK;
}

}  // namespace eagle
