// tree_attention.cu -- tree-masked GQA attention of the flattened draft tree (sm_103a).
//
// Pages: "LLM speculative decoding explained" (hubwiz.com) section 5 -- the flattened tree is
// scored in one target pass and every candidate sees only its ancestors and the context; and
// "(EAGLE 2) EAGLE-2 ..." section "Tree Attention Mask".
//
// Work unit: (layer l, sequence b, KV head g).  Its query block is the G = Hq/Hkv query heads of
// every tree node, row r = node * G + head-in-group, so that all query heads sharing one KV head
// stream the context once.  The context keys are unmasked; the n tree keys form one extra 64-key
// tile whose visibility is the node's ancestor bit mask (one 64-bit word per node).
//
// bf16 kernel: CTA = (unit, 64-row group); 4 warps x 16 query rows; K/V tiles of 64 keys are
// staged in shared memory with cp.async (double buffered, 16-byte chunks XOR-swizzled by key so
// ldmatrix is conflict-free); QK^T and PV use bf16 mma.sync m16n8k16 with fp32 accumulation;
// online softmax in base 2 on the SFU.  The row groups of a unit are adjacent in the grid, so the
// unit's K/V bytes come from HBM once and from L2 for the other groups.
// fp32 kernel: plain FFMA flash attention (16 query rows per CTA, 32-key tiles in shared memory),
// for the fp32 workload and its 1e-4 bar.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "common.cuh"

namespace eagle {

struct AttnTcParams {
    const uint64_t *mask;
    const int32_t *ctx_len;
    __nv_bfloat16 *out;
    int32_t *status;
    int L, B, n, Hq, Hkv, G, S_max, rows, mgroups;
    int HD;
    float scale_log2;
    int splits;
    float *part_o;
    float *part_ml;
};
bool tree_attention_tc_supported(int head_dim, int dtype, int G, int S_max);
eagle_status tree_attention_tc_launch(const AttnTcParams &p, const void *q, const void *k_cache, const void *v_cache,
                                      const void *k_tree, const void *v_tree, cudaStream_t stream);

struct AttnArgs {
    const void *q, *k_cache, *v_cache, *k_tree, *v_tree;
    const int32_t *ctx_len;
    const uint64_t *mask;
    void *out;
    int32_t *status;
    int L, B, n, Hq, Hkv, G, S_max, rows, mgroups;
    float scale_log2;  // softmax scale * log2(e)
    float scale;
};

namespace {

constexpr int kTileKeys = 64;
constexpr int kWarps = 4;
constexpr int kRowsPerCta = 16 * kWarps;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                                  uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of 16-byte chunk `chunk` of key row `key` in a swizzled [64][HD] bf16 tile.
template <int HD>
__device__ __forceinline__ uint32_t tile_off(int key, int chunk) {
    return uint32_t(key * HD * 2 + ((chunk ^ (key & 7)) << 4));
}

// Stage one 64-key tile of K and V (rows `nrows` valid, the rest zero-filled).
template <int HD>
__device__ __forceinline__ void load_tile(uint32_t sk, uint32_t sv, const __nv_bfloat16 *kbase,
                                          const __nv_bfloat16 *vbase, size_t row_stride, int nrows, int tid) {
    constexpr int CPR = HD / 8;  // 16-byte chunks per key row
    constexpr int TOTAL = kTileKeys * CPR;
#pragma unroll
    for (int it = 0; it < TOTAL / (32 * kWarps); ++it) {
        const int cid = tid + it * 32 * kWarps;
        const int key = cid / CPR, ch = cid % CPR;
        const bool ok = key < nrows;
        const size_t goff = (ok ? size_t(key) * row_stride : 0) + size_t(ch) * 8;
        cp_async16(sk + tile_off<HD>(key, ch), kbase + goff, ok ? 16 : 0);
        cp_async16(sv + tile_off<HD>(key, ch), vbase + goff, ok ? 16 : 0);
    }
}

template <int HD>
__global__ void __launch_bounds__(32 * kWarps) tree_attn_bf16_kernel(AttnArgs a) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int KC = HD / 16;  // k16 chunks of the head dim
    constexpr int DT = HD / 8;   // n8 tiles of the head dim
    constexpr int TILE_BYTES = kTileKeys * HD * 2;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int mg = blockIdx.x % a.mgroups;
    const int unit = blockIdx.x / a.mgroups;
    const int g = unit % a.Hkv;
    const int b = (unit / a.Hkv) % a.B;
    const int l = unit / (a.Hkv * a.B);

    const int ctx = a.ctx_len[b];
    if (ctx < 0 || ctx > a.S_max) {
        if (tid == 0 && mg == 0 && g == 0) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
        return;
    }

    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.q);
    const size_t kv_stride = size_t(a.Hkv) * HD;  // between consecutive keys
    const __nv_bfloat16 *kc = static_cast<const __nv_bfloat16 *>(a.k_cache) +
                              ((size_t(l) * a.B + b) * a.S_max * a.Hkv + g) * HD;
    const __nv_bfloat16 *vc = static_cast<const __nv_bfloat16 *>(a.v_cache) +
                              ((size_t(l) * a.B + b) * a.S_max * a.Hkv + g) * HD;
    const __nv_bfloat16 *kt = static_cast<const __nv_bfloat16 *>(a.k_tree) +
                              ((size_t(l) * a.B + b) * a.n * a.Hkv + g) * HD;
    const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(a.v_tree) +
                              ((size_t(l) * a.B + b) * a.n * a.Hkv + g) * HD;

    const uint32_t s_base = smem_u32(smem);
    // stage s: K at s_base + s*2*TILE_BYTES, V right after
    const int ntiles_ctx = (ctx + kTileKeys - 1) / kTileKeys;
    const int ntiles = ntiles_ctx + 1;  // + the tree tile

    auto issue = [&](int t, int stage) {
        const uint32_t sk = s_base + stage * 2 * TILE_BYTES, sv = sk + TILE_BYTES;
        if (t < ntiles_ctx) {
            const int k0 = t * kTileKeys;
            load_tile<HD>(sk, sv, kc + size_t(k0) * kv_stride, vc + size_t(k0) * kv_stride, kv_stride,
                          min(kTileKeys, ctx - k0), tid);
        } else {
            load_tile<HD>(sk, sv, kt, vt, kv_stride, a.n, tid);
        }
        cp_async_commit();
    };
    issue(0, 0);

    // query rows of this warp: r0 = first row; thread rows ra = r0 + lane/4, rb = ra + 8
    const int r0 = mg * kRowsPerCta + warp * 16;
    const int ra = r0 + (lane >> 2), rb = ra + 8;
    const bool va = ra < a.rows, vb = rb < a.rows;
    const int na = va ? ra / a.G : 0, nb = vb ? rb / a.G : 0;
    const int ha = g * a.G + (va ? ra % a.G : 0), hb = g * a.G + (vb ? rb % a.G : 0);
    const size_t qa = va ? (((size_t(l) * a.B + b) * a.n + na) * a.Hq + ha) * HD : 0;
    const size_t qb = vb ? (((size_t(l) * a.B + b) * a.n + nb) * a.Hq + hb) * HD : 0;
    const uint64_t mask_a = va ? a.mask[size_t(b) * a.n + na] : 0ull;
    const uint64_t mask_b = vb ? a.mask[size_t(b) * a.n + nb] : 0ull;

    uint32_t qf[KC][4];
#pragma unroll
    for (int kc2 = 0; kc2 < KC; ++kc2) {
        const int c0 = kc2 * 16 + (lane & 3) * 2;
        qf[kc2][0] = va ? *reinterpret_cast<const uint32_t *>(Q + qa + c0) : 0u;
        qf[kc2][1] = vb ? *reinterpret_cast<const uint32_t *>(Q + qb + c0) : 0u;
        qf[kc2][2] = va ? *reinterpret_cast<const uint32_t *>(Q + qa + c0 + 8) : 0u;
        qf[kc2][3] = vb ? *reinterpret_cast<const uint32_t *>(Q + qb + c0 + 8) : 0u;
    }

    float o[DT][4];
#pragma unroll
    for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    for (int t = 0; t < ntiles; ++t) {
        const int stage = t & 1;
        if (t + 1 < ntiles) {
            issue(t + 1, stage ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint32_t sk = s_base + stage * 2 * TILE_BYTES, sv = sk + TILE_BYTES;
        const bool tree_tile = t >= ntiles_ctx;
        const int kvalid = tree_tile ? a.n : min(kTileKeys, ctx - t * kTileKeys);

        // S = Q K^T for 64 keys: 8 n8 tiles
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kc2 = 0; kc2 < KC; ++kc2) {
#pragma unroll
            for (int nt = 0; nt < 8; nt += 2) {
                const int mi = lane >> 3, rr = lane & 7;
                const int key = (nt + (mi >> 1)) * 8 + rr;
                const int ch = 2 * kc2 + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(sk + tile_off<HD>(key, ch), b0, b1, b2, b3);
                mma_bf16(s[nt], qf[kc2], b0, b1);
                mma_bf16(s[nt + 1], qf[kc2], b2, b3);
            }
        }
        // scale, mask, running max
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = nt * 8 + (lane & 3) * 2 + e;
                bool ok_a = key < kvalid, ok_b = key < kvalid;
                if (tree_tile) {
                    ok_a = ok_a && ((mask_a >> key) & 1ull);
                    ok_b = ok_b && ((mask_b >> key) & 1ull);
                }
                const float xa = ok_a ? s[nt][e] * a.scale_log2 : -INFINITY;
                const float xb = ok_b ? s[nt][2 + e] * a.scale_log2 : -INFINITY;
                s[nt][e] = xa;
                s[nt][2 + e] = xb;
                mx_a = fmaxf(mx_a, xa);
                mx_b = fmaxf(mx_b, xb);
            }
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
        }
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float ref_a = mn_a == -INFINITY ? 0.f : mn_a;
        const float ref_b = mn_b == -INFINITY ? 0.f : mn_b;
        const float alpha_a = fast_exp2(m_a - ref_a), alpha_b = fast_exp2(m_b - ref_b);
        m_a = mn_a;
        m_b = mn_b;
        float sum_a = 0.f, sum_b = 0.f;
        uint32_t pf[4][4];  // P as A fragments: 4 k16 chunks of 16 keys
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float p0 = fast_exp2(s[nt][0] - ref_a), p1 = fast_exp2(s[nt][1] - ref_a);
            const float p2 = fast_exp2(s[nt][2] - ref_b), p3 = fast_exp2(s[nt][3] - ref_b);
            sum_a += p0 + p1;
            sum_b += p2 + p3;
            const int kc2 = nt >> 1, hi = nt & 1;
            pf[kc2][hi * 2 + 0] = pack_bf16(p0, p1);
            pf[kc2][hi * 2 + 1] = pack_bf16(p2, p3);
        }
        l_a = l_a * alpha_a + sum_a;
        l_b = l_b * alpha_b + sum_b;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
            o[dt][0] *= alpha_a;
            o[dt][1] *= alpha_a;
            o[dt][2] *= alpha_b;
            o[dt][3] *= alpha_b;
        }
        // O += P V
#pragma unroll
        for (int kc2 = 0; kc2 < 4; ++kc2) {
#pragma unroll
            for (int dt = 0; dt < DT; dt += 2) {
                const int mi = lane >> 3, rr = lane & 7;
                const int key = kc2 * 16 + (mi & 1) * 8 + rr;
                const int ch = dt + (mi >> 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(sv + tile_off<HD>(key, ch), b0, b1, b2, b3);
                mma_bf16(o[dt], pf[kc2], b0, b1);
                mma_bf16(o[dt + 1], pf[kc2], b2, b3);
            }
        }
        __syncthreads();  // the stage is refilled by the next iteration's issue
    }

    // normalise and store (row sums over the quad)
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
    }
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
    const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
    __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(a.out);
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
        const int c0 = dt * 8 + (lane & 3) * 2;
        if (va) *reinterpret_cast<uint32_t *>(O + qa + c0) = pack_bf16(o[dt][0] * inv_a, o[dt][1] * inv_a);
        if (vb) *reinterpret_cast<uint32_t *>(O + qb + c0) = pack_bf16(o[dt][2] * inv_b, o[dt][3] * inv_b);
    }
}

// fp32: a CTA per (unit, block of kF32Rows query rows), 256 threads.  The unit's keys (its
// context, then the n tree keys) stream through shared memory in tiles of kF32Keys, the next
// tile's loads in flight (in registers) while the current one is used; thread t owns
// query row t / 16 of the block: two of the tile's scores (keys t % 16 and t % 16 + 16, full dot
// products from shared memory) and HD / 16 output columns (t % 16 + 16 c).  The 16 threads of a
// row are one half-warp, so the row's online softmax (running max, rescale, running sum) meets by
// shuffles and its probabilities pass through shared memory under a warp barrier only.  Keys that
// a row does not see score -inf; the rows of absent keys are zero in shared memory, so whatever a
// cache position past the context holds never reaches an output.
constexpr int kF32Rows = 16;
constexpr int kF32Keys = 32;
constexpr int kF32Threads = 256;

template <int HD>
__global__ void __launch_bounds__(kF32Threads) tree_attn_f32_kernel(AttnArgs a) {
    pdl_wait();
    pdl_launch_next();
    constexpr int NO = HD / 16;  // output columns per thread
    __shared__ float sQ[kF32Rows][HD + 1];  // padded: the two half-warps' rows sit in different banks
    __shared__ float sK[kF32Keys][HD + 1];  // padded: the 16 keys a half-warp reads sit in distinct banks
    __shared__ float sV[kF32Keys][HD];
    __shared__ float sP[kF32Rows][kF32Keys + 1];
    const int tid = threadIdx.x;
    const int rblocks = (a.rows + kF32Rows - 1) / kF32Rows;
    const int unit = blockIdx.x / rblocks, rb = blockIdx.x % rblocks;
    const int g = unit % a.Hkv;
    const int b = (unit / a.Hkv) % a.B;
    const int l = unit / (a.Hkv * a.B);
    const int ctx = a.ctx_len[b];
    if (ctx < 0 || ctx > a.S_max) {
        if (tid == 0 && g == 0 && rb == 0) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
        return;  // uniform for the CTA
    }
    const float *Q = static_cast<const float *>(a.q);
    const float *kc = static_cast<const float *>(a.k_cache) + ((size_t(l) * a.B + b) * a.S_max * a.Hkv + g) * HD;
    const float *vc = static_cast<const float *>(a.v_cache) + ((size_t(l) * a.B + b) * a.S_max * a.Hkv + g) * HD;
    const float *kt = static_cast<const float *>(a.k_tree) + ((size_t(l) * a.B + b) * a.n * a.Hkv + g) * HD;
    const float *vt = static_cast<const float *>(a.v_tree) + ((size_t(l) * a.B + b) * a.n * a.Hkv + g) * HD;
    const size_t stride = size_t(a.Hkv) * HD;  // between consecutive keys of one KV head

    // the block's query rows, pre-scaled (row r: node r / G, query head g G + r % G)
    const int r0 = rb * kF32Rows;
    for (int i = tid; i < kF32Rows * (HD / 4); i += kF32Threads) {
        const int rr = i / (HD / 4), c4 = i % (HD / 4), r = r0 + rr;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < a.rows) {
            const size_t qo = (((size_t(l) * a.B + b) * a.n + r / a.G) * a.Hq + g * a.G + r % a.G) * HD;
            v = reinterpret_cast<const float4 *>(Q + qo)[c4];
            v.x *= a.scale;
            v.y *= a.scale;
            v.z *= a.scale;
            v.w *= a.scale;
        }
        sQ[rr][4 * c4] = v.x;
        sQ[rr][4 * c4 + 1] = v.y;
        sQ[rr][4 * c4 + 2] = v.z;
        sQ[rr][4 * c4 + 3] = v.w;
    }
    const int orow = tid >> 4, sub = tid & 15;
    const int r = r0 + orow;
    const bool rvalid = r < a.rows;
    const uint64_t tmask = rvalid ? a.mask[size_t(b) * a.n + r / a.G] : 0ull;
    float o[NO];
#pragma unroll
    for (int c = 0; c < NO; ++c) o[c] = 0.f;
    float m = -INFINITY, lsum = 0.f;
    const int nk = ctx + a.n;  // the context's keys, then the tree's
    // this thread's share of a tile: NL float4 of K and of V (zero past the unit's keys)
    constexpr int NL = kF32Keys * (HD / 4) / kF32Threads;
    float4 kr[NL], vr[NL];
    auto load_tile = [&](int j0) {
#pragma unroll
        for (int u = 0; u < NL; ++u) {
            const int i = tid + u * kF32Threads;
            const int jj = i / (HD / 4), c4 = i % (HD / 4), j = j0 + jj;
            kr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            vr[u] = kr[u];
            if (j < ctx) {
                kr[u] = reinterpret_cast<const float4 *>(kc + size_t(j) * stride)[c4];
                vr[u] = reinterpret_cast<const float4 *>(vc + size_t(j) * stride)[c4];
            } else if (j < nk) {
                kr[u] = reinterpret_cast<const float4 *>(kt + size_t(j - ctx) * stride)[c4];
                vr[u] = reinterpret_cast<const float4 *>(vt + size_t(j - ctx) * stride)[c4];
            }
        }
    };
    load_tile(0);
    for (int j0 = 0; j0 < nk; j0 += kF32Keys) {
        __syncthreads();  // the previous tile is consumed (and, the first time, sQ is written)
#pragma unroll
        for (int u = 0; u < NL; ++u) {
            const int i = tid + u * kF32Threads;
            const int jj = i / (HD / 4), c4 = i % (HD / 4);
            sK[jj][4 * c4] = kr[u].x;
            sK[jj][4 * c4 + 1] = kr[u].y;
            sK[jj][4 * c4 + 2] = kr[u].z;
            sK[jj][4 * c4 + 3] = kr[u].w;
            *reinterpret_cast<float4 *>(&sV[jj][4 * c4]) = vr[u];
        }
        __syncthreads();
        if (j0 + kF32Keys < nk) load_tile(j0 + kF32Keys);  // in flight while this tile is used
        // two scores of this thread's row: keys sub and sub + 16 of the tile (four partial sums
        // a dot product, so its chain is a quarter as long)
        float s2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int jj = sub + 16 * h, j = j0 + jj;
            const bool vis = rvalid && (j < ctx || (j < nk && ((tmask >> (j - ctx)) & 1ull)));
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int d = 0; d < HD; d += 4) {
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = fmaf(sQ[orow][d + e], sK[jj][d + e], acc[e]);
            }
            s2[h] = vis ? (acc[0] + acc[1]) + (acc[2] + acc[3]) : -INFINITY;
        }
        // online softmax over the row's half-warp
        float tmx = fmaxf(s2[0], s2[1]);
#pragma unroll
        for (int x = 8; x > 0; x >>= 1) tmx = fmaxf(tmx, __shfl_xor_sync(0xffffffffu, tmx, x));
        const float mn = fmaxf(m, tmx);
        const float alpha = mn == -INFINITY ? 1.f : expf(m - mn);  // m = -inf: nothing to rescale
        const float p0 = s2[0] == -INFINITY ? 0.f : expf(s2[0] - mn);
        const float p1 = s2[1] == -INFINITY ? 0.f : expf(s2[1] - mn);
        float ps = p0 + p1;
#pragma unroll
        for (int x = 8; x > 0; x >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, x);
        lsum = lsum * alpha + ps;
        m = mn;
        sP[orow][sub] = p0;
        sP[orow][sub + 16] = p1;
        __syncwarp();  // the row's probabilities are written by its own half-warp
#pragma unroll
        for (int c = 0; c < NO; ++c) o[c] *= alpha;
#pragma unroll 8
        for (int jj = 0; jj < kF32Keys; ++jj) {
            const float p = sP[orow][jj];
#pragma unroll
            for (int c = 0; c < NO; ++c) o[c] = fmaf(p, sV[jj][sub + 16 * c], o[c]);
        }
        __syncwarp();  // sP is rewritten by the next tile
    }
    if (!rvalid) return;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    float *O = static_cast<float *>(a.out) +
               (((size_t(l) * a.B + b) * a.n + r / a.G) * a.Hq + g * a.G + r % a.G) * HD;
#pragma unroll
    for (int c = 0; c < NO; ++c) O[sub + 16 * c] = o[c] * inv;
}

template <int HD>
eagle_status launch_bf16(const AttnArgs &a, cudaStream_t stream) {
    constexpr size_t smem = size_t(2) * 2 * kTileKeys * HD * 2;  // 2 stages x (K + V)
    static std::atomic<uint64_t> ready{0};
    if (once_per_device(ready, [&] {
            return cudaFuncSetAttribute(tree_attn_bf16_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(smem));
        }) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    const long grid = long(a.L) * a.B * a.Hkv * a.mgroups;
    if (launch_pdl(tree_attn_bf16_kernel<HD>, dim3(unsigned(grid)), dim3(32 * kWarps), smem, stream, 1u, a) !=
        cudaSuccess)
        return EAGLE_ERR_CUDA;
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

template <int HD>
eagle_status launch_f32(const AttnArgs &a, cudaStream_t stream) {
    const long grid = long(a.L) * a.B * a.Hkv * ((a.rows + kF32Rows - 1) / kF32Rows);
    if (launch_pdl(tree_attn_f32_kernel<HD>, dim3(unsigned(grid)), dim3(kF32Threads), 0, stream, 1u, a) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}


}  // namespace

// Context split of the tensor-core kernel: when the (layer, sequence, KV head, row group) units
// fill less than half of the GPU's SMs (a draft model's single layer, one sequence), each unit's
// context tiles are shared among several CTAs whose partial results a merge kernel combines
// exactly; the workspace then holds the partials.
int attn_tc_splits(const eagle_attn_cfg &c) {
    if (c.dtype != EAGLE_DTYPE_BF16 || (c.head_dim != 128 && c.head_dim != 64) || c.heads_kv < 1 || c.heads_q % c.heads_kv ||
        c.heads_q / c.heads_kv > 128)
        return 1;
    const long rows = long(c.heads_q / c.heads_kv) * c.nodes;
    const long cta_rows = 2L * attn_tc_rows_per_mtile(c.heads_q / c.heads_kv);
    const long units = long(c.layers) * c.batch * c.heads_kv * ((rows + cta_rows - 1) / cta_rows);
    const long sms = device_sm_count();
    if (units * 2 > sms) return 1;
    const long nctx = (long(c.max_seq) + 127) / 128;
    long s = sms / units;
    if (s > nctx / 2) s = nctx / 2;  // at least two tiles a split: the partials and the merge stay small
    if (s > 32) s = 32;
    return s < 2 ? 1 : int(s);
}

size_t attn_tc_partial_rows(const eagle_attn_cfg &c, int splits) {
    const long rows = long(c.heads_q / c.heads_kv) * c.nodes;
    const long cta_rows = 2L * attn_tc_rows_per_mtile(c.heads_q / c.heads_kv);
    return size_t(c.layers) * c.batch * c.heads_kv * ((rows + cta_rows - 1) / cta_rows) * splits * 256;
}

size_t tree_attention_workspace_bytes(const eagle_attn_cfg &c) {
    const int splits = attn_tc_splits(c);
    if (splits == 1) return kWsHeader;
    const size_t prow = attn_tc_partial_rows(c, splits);
    return kWsHeader + align_up(prow * 2 * sizeof(float), 256) + align_up(prow * 128 * sizeof(float), 256);
}

eagle_status tree_attention_launch(const eagle_attn_cfg &c, const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *ctx_len, const void *k_tree, const void *v_tree,
                                   const uint64_t *mask, void *out, void *ws, cudaStream_t stream) {
    AttnArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_tree = k_tree;
    a.v_tree = v_tree;
    a.ctx_len = ctx_len;
    a.mask = mask;
    a.out = out;
    a.status = static_cast<int32_t *>(ws);
    a.L = c.layers;
    a.B = c.batch;
    a.n = c.nodes;
    a.Hq = c.heads_q;
    a.Hkv = c.heads_kv;
    a.G = c.heads_q / c.heads_kv;
    a.S_max = c.max_seq;
    a.rows = a.G * a.n;
    a.mgroups = (a.rows + kRowsPerCta - 1) / kRowsPerCta;
    a.scale = c.scale > 0.f ? c.scale : 1.f / sqrtf(float(c.head_dim));
    a.scale_log2 = a.scale * kLog2e;
    if (c.dtype == EAGLE_DTYPE_BF16) {
        if (tree_attention_tc_supported(c.head_dim, c.dtype, a.G, c.max_seq)) {
            AttnTcParams tp;
            tp.mask = mask;
            tp.ctx_len = ctx_len;
            tp.out = static_cast<__nv_bfloat16 *>(out);
            tp.status = a.status;
            tp.L = a.L;
            tp.B = a.B;
            tp.n = a.n;
            tp.Hq = a.Hq;
            tp.Hkv = a.Hkv;
            tp.G = a.G;
            tp.S_max = a.S_max;
            tp.rows = a.rows;
            tp.HD = c.head_dim;
            tp.mgroups = (a.rows + 2 * attn_tc_rows_per_mtile(a.G) - 1) / (2 * attn_tc_rows_per_mtile(a.G));
            tp.scale_log2 = a.scale_log2;
            tp.splits = attn_tc_splits(c);
            tp.part_ml = nullptr;
            tp.part_o = nullptr;
            if (tp.splits > 1) {
                unsigned char *w = static_cast<unsigned char *>(ws);
                const size_t prow = attn_tc_partial_rows(c, tp.splits);
                tp.part_ml = reinterpret_cast<float *>(w + kWsHeader);
                tp.part_o = reinterpret_cast<float *>(w + kWsHeader + align_up(prow * 2 * sizeof(float), 256));
            }
            const eagle_status st = tree_attention_tc_launch(tp, q, k_cache, v_cache, k_tree, v_tree, stream);
            if (st != EAGLE_ERR_UNSUPPORTED) return st;
        }
        return c.head_dim == 128 ? launch_bf16<128>(a, stream) : launch_bf16<64>(a, stream);
    }
    return c.head_dim == 128 ? launch_f32<128>(a, stream) : launch_f32<64>(a, stream);
}

}  // namespace eagle
