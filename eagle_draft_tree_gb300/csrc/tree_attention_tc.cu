// tree_attention_tc.cu -- tree-masked GQA attention on the 5th-generation tensor cores (sm_103a).
//
// Pages: "LLM speculative decoding explained" (hubwiz.com) section 5 -- the flattened tree is
// scored in one target pass and every candidate sees only its ancestors and the context; and
// "(EAGLE 2) EAGLE-2 ..." section "Tree Attention Mask".
//
// One CTA = one (layer, sequence, KV head) unit and up to two M-tiles of its query block (row
// r = node * G + head-in-group); an M-tile holds floor(128 / G) whole nodes, all 128 TMEM lanes
// when G divides 128, else G floor(128 / G) of them and a few padding lanes that nothing reads.
// The context streams through in 128-key tiles; the n <= 64 tree keys form one last tile whose
// visibility is the node's ancestor bit mask.
//
//   warp 0     TMA producer: Q once (two 64-column halves per M-tile), then K and V tiles (one
//              4-D box per tile: 128 keys x both 64-dim halves, 128B-swizzled) through a 2-stage K
//              ring and a 3-stage V ring, in the order K(j), V(j), each as soon as its stage is free.
//   warp 1     the MMA issuer for both M-tiles (a whole converged warp, one elected lane issues),
//              in a fixed order: S_0(0), S_1(0), then per tile j: O_0 += P_0(j) V(j), S_0(j + 1),
//              O_1 += P_1(j) V(j), S_1(j + 1).  P_t (bf16 pairs, written by the softmax over the
//              first 64 columns of S_t) is the A operand, read from tensor memory; S_t(j + 1) is
//              issued right behind the PV that reads P_t(j) (the MMAs of one thread execute in
//              order), so a softmax warpgroup restarts as soon as its own PV and next QK^T are
//              through, and the two warpgroups settle half a period apart.
//   warps 4-11 two softmax warpgroups, one per M-tile, one thread per query row, each tile in two
//              64-key chunks: tcgen05.ld, mask, base-2 online softmax with lazy rescaling (O in
//              TMEM is rescaled only when the running max grows by more than 8, i.e. P <= 2^8; the
//              commit of S_t(j) covers PV_t(j - 1), so O_t is at rest then), P to TMEM, and the
//              final O / l epilogue.  M-tile 0's warpgroup also zeroes the V rows past the last
//              visible key of the ragged context tile and of the tree tile before their PV (P is 0
//              there, but 0 x NaN would not be).
//
// Every mbarrier wait gives up after one second; a wait that runs out records EAGLE_ERR_TIMEOUT in
// the status word, raises a CTA-wide abort flag that ends every role's loop, and the CTA still
// drains its issued copies and MMAs (bounded) before releasing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace eagle {

struct AttnTcParams {  // same layout as the declaration in tree_attention.cu
    const uint64_t *mask;
    const int32_t *ctx_len;
    __nv_bfloat16 *out;
    int32_t *status;
    int L, B, n, Hq, Hkv, G, S_max, rows, mgroups;
    int HD;         // head dimension: 128, or 64 (run as 128 with a zero upper half)
    float scale_log2;
    int splits;     // context splits per unit (1: each CTA writes its rows' output itself)
    float *part_o;  // splits > 1: [unit][split][mgroup][256 rows][128] unnormalised partial O
    float *part_ml; // splits > 1: [unit][split][mgroup][256 rows][2] (max in base-2 units, sum)
};

namespace {

constexpr int kThreads = 384;
constexpr int kNkv = 128;                   // keys per tile
constexpr int kKStages = 2;                 // K tiles are released as soon as both QK^T have read them
constexpr int kVStages = 3;                 // V tiles are held until both PV, later in the tile's life
constexpr uint32_t kHalf = kNkv * 128;      // one 64-dim half of a K or V tile: 128 rows x 128 B
constexpr uint32_t kTileBytes = 2 * kHalf;  // a K (or V) tile: both halves
constexpr uint32_t kQHalf = 128 * 128;      // 128 rows x 128 B
constexpr uint32_t kQTile = 2 * kQHalf;
constexpr uint32_t kOffK = 2 * kQTile;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kSmemBytes = kOffV + kVStages * kTileBytes;  // 224 KB
// TMEM columns: O_0, O_1 (128 each) | S_0, S_1 (128 fp32 each; P_t over the first 64 of S_t)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;

__device__ __forceinline__ uint32_t sa(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    // start >> 4 [0,14), LBO >> 4 [16,30), SBO >> 4 [32,46), version 1 at bit 46, 128B swizzle (2)
    return uint64_t((addr >> 4) & 0x3FFF) | (uint64_t((lbo >> 4) & 0x3FFF) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFF) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
// kind::f16 instruction descriptor: D f32, A and B bf16, K-major A, B K- or MN-major
constexpr uint32_t idesc(int M, int N, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(b_mn) << 16) | (uint32_t(N >> 3) << 17) |
           (uint32_t(M >> 4) << 24);
}
constexpr uint32_t kIdescQK = idesc(128, kNkv, 0);  // N = 128 keys
constexpr uint32_t kIdescQK64 = idesc(128, 64, 0);  // the tree tile: N = 64 keys (a tree has <= 64 nodes)
constexpr int kTreeKeys = 64;
constexpr uint32_t kIdescPV = idesc(128, 128, 1);  // A = P from TMEM, B = V MN-major

// The MMA issuer is a whole converged warp; one lane, picked by elect.sync, issues each operation
// (issuing from a converged warp is faster than from one lane of a divergent branch).
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
// A from TMEM (K-major, two bf16 per 32-bit column), B from shared memory
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(sa(bar))
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(bar)) : "memory");
}
// One 4-D box: both 64-dim halves of kNkv rows of one KV head; lands as [half][row][128 B].  The
// KV cache is read once per call and is larger than L2, so its lines are marked evict-first:
// the L2 keeps what the other kernels of a round reuse (their code, the draft rows, the tree).
__device__ __forceinline__ void tma_kv(const CUtensorMap *map, void *dst, uint64_t *bar, int row, int head,
                                       uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4, %5}], [%6], %7;" ::"r"(sa(dst)),
        "l"(map), "r"(0), "r"(row), "r"(0), "r"(head), "r"(sa(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_3d(const CUtensorMap *map, void *dst, uint64_t *bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(sa(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(sa(bar))
        : "memory");
}
// 16 consecutive TMEM columns of this warp's 32 lanes (no wait)
__device__ __forceinline__ void tld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tst16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
__device__ __forceinline__ void tst_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Two floats in one 64-bit register pair, for the f32x2 arithmetic of sm_100-class SMs.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float f2_lo(uint64_t r) {
    float a;
    asm("{\n .reg .f32 x;\n mov.b64 {%0, x}, %1;\n}" : "=f"(a) : "l"(r));
    return a;
}
__device__ __forceinline__ float f2_hi(uint64_t r) {
    float b;
    asm("{\n .reg .f32 x;\n mov.b64 {x, %0}, %1;\n}" : "=f"(b) : "l"(r));
    return b;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

struct Bars {
    uint64_t q_full;
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t v_clean[2];  // V rows past the last visible key zeroed: [0] ragged context tile, [1] tree tile
    uint64_t s_full[2];   // [M-tile]: QK^T of the current tile landed (and every MMA issued before it)
    uint64_t p_full[2];   // [M-tile]: P of the current tile written over S_t
    uint64_t o_done[2];   // [M-tile]: the last PV completed
    uint64_t drain;       // every MMA of the issuing warp completed
};

// Bounded wait; gives up (and raises the abort flag) when the CTA aborted or the deadline passed.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *status) {
    Deadline d;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255) == 255 && *abort_flag) return false;
        if (d.passed(it)) break;
    }
    *abort_flag = 1;
    set_status(status, EAGLE_ERR_TIMEOUT);
    return false;
}

// Warp-uniform bounded wait: every lane polls and the warp agrees by vote, so the warp never
// diverges (a lane-0-only polling loop costs several hundred cycles to reconverge even when the
// phase has long completed; this form costs a few dozen).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int32_t *status) {
    Deadline d;
    for (uint32_t it = 0;; ++it) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if ((it & 255) == 255 && __any_sync(0xffffffffu, *abort_flag != 0)) return false;
        if (d.passed_warp(it)) break;
    }
    if ((threadIdx.x & 31) == 0) {
        *abort_flag = 1;
        set_status(status, EAGLE_ERR_TIMEOUT);
    }
    __syncwarp();
    return false;
}

// Rescale 128 TMEM columns of this warp's 32 lanes (a row of O) by alpha.
__device__ __forceinline__ void tmem_scale128(uint32_t taddr, float alpha) {
#pragma unroll
    for (int cc = 0; cc < 128; cc += 16) {
        uint32_t o[16];
        tld16(taddr + cc, o);
        tld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tst16(taddr + cc, o);
    }
}

// kSplit: the unit's context is shared among p.splits CTAs, each writing a partial result for
// tree_attn_merge_kernel (a separate instance, so the unsplit kernel carries none of it).
template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap ktmap,
                        const __grid_constant__ CUtensorMap vtmap, AttnTcParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Bars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    pdl_wait();
    pdl_launch_next();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int splits = kSplit ? p.splits : 1;
    const int mg = blockIdx.x % p.mgroups;
    const int split = kSplit ? (blockIdx.x / p.mgroups) % splits : 0;
    const int unit = blockIdx.x / (p.mgroups * splits);
    const int g = unit % p.Hkv;
    const int b = (unit / p.Hkv) % p.B;
    const int l = unit / (p.Hkv * p.B);
    const int ctx = p.ctx_len[b];  // in flight during the set-up below, which does not depend on it
    if (tid == 0) {
        s_abort = 0;
        mbar_init(&bars.q_full, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars.v_clean[t], 4);
            mbar_init(&bars.s_full[t], 1);
            mbar_init(&bars.p_full[t], 4);
            mbar_init(&bars.o_done[t], 1);
        }
        mbar_init(&bars.drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sa(&s_tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int *abort_flag = &s_abort;
    // A context length outside [0, S_max], or (context split) a split with no tile: uniform exits
    // for the CTA, which give back its TMEM.
    const bool bad_ctx = ctx < 0 || ctx > p.S_max;
    const int ctxv = bad_ctx ? 0 : ctx;
    const int npt = 128 / p.G, rpt = npt * p.G;            // nodes and query rows of an M-tile
    const int row0 = mg * 2 * rpt;                         // first query row of this CTA
    const int tm = min(2, (p.rows - row0 + rpt - 1) / rpt);  // M-tiles in this CTA (1 or 2)
    const int nctx = (ctxv + kNkv - 1) / kNkv;           // context tiles
    const int jtail = (ctxv % kNkv) ? nctx - 1 : -1;     // the ragged context tile, if any
    // This CTA's share of the unit's tiles: context tiles [c0, c1), and the tree tile in the last
    // split.  Stages, phases and the first-tile test count local tiles j = 0 .. ntiles - 1; the
    // coordinates and the masking use the global tile gtile(j).
    const int tps = kSplit ? (nctx + splits - 1) / splits : nctx;
    const int c0 = kSplit ? min(split * tps, nctx) : 0, c1 = kSplit ? min(c0 + tps, nctx) : nctx;
    const bool has_tree = !kSplit || split == splits - 1;
    const int ntiles = (c1 - c0) + (has_tree ? 1 : 0);
    auto gtile = [&](int j) { return kSplit ? (j < c1 - c0 ? c0 + j : nctx) : j; };
    const size_t pbase = (size_t(unit * splits + split) * p.mgroups + mg) * 256;  // partial rows
    if (bad_ctx || (kSplit && ntiles == 0)) {
        if (bad_ctx) {
            if (tid == 0 && mg == 0 && g == 0) set_status(p.status, EAGLE_ERR_DEVICE_INPUT);
        } else {  // an empty partial
            for (int i = tid; i < 256; i += kThreads) {
                p.part_ml[(pbase + i) * 2] = -INFINITY;
                p.part_ml[(pbase + i) * 2 + 1] = 0.f;
            }
        }
        if (warp == 1)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
        return;
    }

    int k_issued = 0, v_issued = 0;  // producer: K / V tiles whose copies were issued
    if (warp == 0) {
        // ---------------- TMA producer: two rings, issued whenever a stage is free ----------------
        if (lane == 0) {
            const int zq = (l * p.B + b) * p.n + row0 / p.G;  // first node of this CTA's rows
            // an M-tile's box is rpt rows high (rows rpt .. 127 of its buffer are padding whose
            // scores and outputs no row reads)
            mbar_expect_tx(&bars.q_full, uint32_t(tm) * 2u * uint32_t(rpt) * 128u);
            for (int t = 0; t < tm; ++t)
                for (int h = 0; h < 2; ++h)
                    tma_3d(&qmap, sm + t * kQTile + h * kQHalf, &bars.q_full, 64 * h, g * p.G, zq + t * npt);
            const int zc = (l * p.B + b) * p.S_max;
            const int zt = (l * p.B + b) * p.n;
            const uint64_t pol = l2_evict_first_policy();
            // fixed order K(j), V(j); each waits (blocking) for its stage's previous tile to be released
            for (int j = 0; j < ntiles; ++j) {
                const int sk = j % kKStages, sv = j % kVStages;
                if (j >= kKStages && !wait_or_abort(&bars.k_empty[sk], ((j / kKStages) - 1) & 1, abort_flag, p.status))
                    break;
                const int jg = gtile(j);
                mbar_expect_tx(&bars.k_full[sk], kTileBytes);
                tma_kv(jg == nctx ? &ktmap : &kmap, sm + kOffK + sk * kTileBytes, &bars.k_full[sk],
                       jg == nctx ? zt : zc + jg * kNkv, g, pol);
                ++k_issued;
                if (j >= kVStages && !wait_or_abort(&bars.v_empty[sv], ((j / kVStages) - 1) & 1, abort_flag, p.status))
                    break;
                mbar_expect_tx(&bars.v_full[sv], kTileBytes);
                tma_kv(jg == nctx ? &vtmap : &vmap, sm + kOffV + sv * kTileBytes, &bars.v_full[sv],
                       jg == nctx ? zt : zc + jg * kNkv, g, pol);
                ++v_issued;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer for both M-tiles, in a fixed order ----------------------------
        bool ok = warp_wait(&bars.q_full, 0, abort_flag, p.status);
        tc_fence_after();
        // S_t(j) = Q_t K(j)^T into S_t (N = 128 keys; the tree tile's 64 first keys only, as a
        // tree has at most 64 nodes)
        auto issue_s = [&](int t, int j) {
            const uint32_t qbase = sa(sm + t * kQTile);
            const uint32_t kbase = sa(sm + kOffK + (j % kKStages) * kTileBytes);
            const uint32_t dS = tmem + kColS + t * 128;
            const uint32_t id = gtile(j) == nctx ? kIdescQK64 : kIdescQK;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * kQHalf + (kk & 3) * 32;
                const uint32_t offk = (kk >> 2) * kHalf + (kk & 3) * 32;
                umma(dS, sdesc(qbase + off, 16, 1024), sdesc(kbase + offk, 16, 1024), id, kk > 0);
            }
            umma_commit(&bars.s_full[t]);
        };
        // O_t += P_t(j) V(j), P_t read from the first 64 columns of S_t (the tree tile: its first
        // 64 keys, P over the first 32 columns)
        auto issue_pv = [&](int t, int j) {
            const uint32_t vbase = sa(sm + kOffV + (j % kVStages) * kTileBytes);
            const uint32_t aP = tmem + kColS + t * 128, dO = tmem + t * 128;
            const int nk = (gtile(j) == nctx ? kTreeKeys : kNkv) / 16;
#pragma unroll
            for (int kk = 0; kk < kNkv / 16; ++kk)
                if (kk < nk)
                    umma_ts(dO, aP + kk * 8, sdesc(vbase + kk * 2048, kHalf, 1024), kIdescPV,
                            (j > 0 || kk > 0) ? 1u : 0u);
        };
        if (ok && (ok = warp_wait(&bars.k_full[0], 0, abort_flag, p.status))) {
            tc_fence_after();
            issue_s(0, 0);
            if (tm > 1) issue_s(1, 0);
            umma_commit(&bars.k_empty[0]);
        }
        for (int j = 0; ok && j < ntiles; ++j) {
            const int sv = j % kVStages, jn = j + 1;
            // V(j) landed (and cleaned, for the ragged and the tree tile), P_0(j) written
            ok = warp_wait(&bars.v_full[sv], (j / kVStages) & 1, abort_flag, p.status) &&
                 (gtile(j) != jtail || warp_wait(&bars.v_clean[0], 0, abort_flag, p.status)) &&
                 (gtile(j) != nctx || warp_wait(&bars.v_clean[1], 0, abort_flag, p.status)) &&
                 warp_wait(&bars.p_full[0], j & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_pv(0, j);
            if (jn < ntiles) {
                if (!(ok = warp_wait(&bars.k_full[jn % kKStages], (jn / kKStages) & 1, abort_flag, p.status))) break;
                tc_fence_after();
                issue_s(0, jn);  // overwrites P_0(j) after the PV just issued has read it
            }
            if (tm > 1) {
                if (!(ok = warp_wait(&bars.p_full[1], j & 1, abort_flag, p.status))) break;
                tc_fence_after();
                issue_pv(1, j);
            }
            umma_commit(&bars.v_empty[sv]);  // both PVs of tile j have read V(j)
            if (jn < ntiles) {
                if (tm > 1) issue_s(1, jn);
                umma_commit(&bars.k_empty[jn % kKStages]);  // both QK^T of tile j + 1 have read K(j + 1)
            } else {
                umma_commit(&bars.o_done[0]);
                umma_commit(&bars.o_done[1]);
            }
        }
        // drain: every MMA issued by this warp has completed once `drain` completes
        umma_commit(&bars.drain);
        mbar_warp_wait_bounded(&bars.drain, 0);
    } else if (warp >= 4 && warp - 4 < 4 * tm) {
        // ---------------- softmax warpgroup t ----------------
        const int t = (warp - 4) >> 2;
        const int wq = warp & 3;  // TMEM lane quarter of this warp
        const int rho = wq * 32 + lane;
        const int r = row0 + t * rpt + rho;
        const bool valid = rho < rpt && r < p.rows;
        const int node = valid ? r / p.G : 0;
        const int gh = valid ? r % p.G : 0;
        const uint64_t tmask = valid ? p.mask[size_t(b) * p.n + node] : 0ull;
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + kColS + t * 128;  // this row's S (P over its first 64 columns)
        const uint32_t tO = tmem + lane_off + t * 128;          // this row's O columns
        const float c = p.scale_log2;
        float m_raw = -INFINITY;  // reference max in raw score units (P = 2^((s - m_raw) c))
        float l_sum = 0.f;
        bool ok = true;
        float sv[64];
        uint32_t pk[32];
        for (int j = 0; j < ntiles; ++j) {
            // S_t(j) landed; its commit also covers PV_t(j - 1), so O_t is at rest
            if (!warp_wait(&bars.s_full[t], j & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int jg = gtile(j);
            const bool tree = jg == nctx;
            const int kvalid = tree ? p.n : min(kNkv, ctx - jg * kNkv);
            float tile_sum = 0.f;
#pragma unroll 1
            for (int q = 0; q < (tree ? 1 : 2); ++q) {  // 64-key chunks (the tree tile has one)
                {
                    uint32_t raw[64];
                    uint32_t (&r0)[16] = *reinterpret_cast<uint32_t(*)[16]>(raw);
                    uint32_t (&r1)[16] = *reinterpret_cast<uint32_t(*)[16]>(raw + 16);
                    uint32_t (&r2)[16] = *reinterpret_cast<uint32_t(*)[16]>(raw + 32);
                    uint32_t (&r3)[16] = *reinterpret_cast<uint32_t(*)[16]>(raw + 48);
                    tld16(tS + q * 64, r0);
                    tld16(tS + q * 64 + 16, r1);
                    tld16(tS + q * 64 + 32, r2);
                    tld16(tS + q * 64 + 48, r3);
                    tld_wait();
#pragma unroll
                    for (int cc = 0; cc < 64; ++cc) sv[cc] = __uint_as_float(raw[cc]);
                }
                // masking: only the ragged context tile and the tree tile have invisible keys (a
                // masked score is replaced, so whatever the fetched K row held is irrelevant)
                const int hv = kvalid - q * 64;
                if (tree || hv < 64) {
                    const int hc = min(max(hv, 0), 64);
                    uint32_t vlo = hc >= 32 ? ~0u : ((1u << hc) - 1u);
                    uint32_t vhi = hc >= 64 ? ~0u : (hc <= 32 ? 0u : ((1u << (hc - 32)) - 1u));
                    if (tree && q == 0) {  // tree keys are keys 0 .. n - 1 <= 63
                        vlo &= uint32_t(tmask);
                        vhi &= uint32_t(tmask >> 32);
                    }
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        if (!((vlo >> cc) & 1u)) sv[cc] = -INFINITY;
                        if (!((vhi >> cc) & 1u)) sv[cc + 32] = -INFINITY;
                    }
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 4) {
                    mx0 = fmaxf(mx0, sv[cc]);
                    mx1 = fmaxf(mx1, sv[cc + 1]);
                    mx2 = fmaxf(mx2, sv[cc + 2]);
                    mx3 = fmaxf(mx3, sv[cc + 3]);
                }
                const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                // lazy rescale: the reference moves only when the max exceeds it by more than 8 in
                // base-2 units, so every P stays below 2^8.  The TMEM accesses below are warp-wide
                // (.sync.aligned), so the warp enters together when any row needs it; the other
                // rows keep their reference and scale by 1.
                const bool moves = m_raw == -INFINITY ? mx != -INFINITY : (mx - m_raw) * c > 8.f;
                if (__any_sync(0xffffffffu, moves)) {
                    const float alpha = !moves ? 1.f : m_raw == -INFINITY ? 0.f : fast_exp2((m_raw - mx) * c);
                    if (moves) m_raw = mx;
                    if (j > 0) tmem_scale128(tO, alpha);  // O_t: tiles < j
                    if (q == 1) {  // P of chunk 0 was computed against the old reference
                        uint32_t q0[16], q1[16];
                        tst_wait();
                        tld16(tS, q0);
                        tld16(tS + 16, q1);
                        tld_wait();
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float2 f0 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&q0[e]));
                            float2 f1 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&q1[e]));
                            __nv_bfloat162 g0 = __floats2bfloat162_rn(f0.x * alpha, f0.y * alpha);
                            __nv_bfloat162 g1 = __floats2bfloat162_rn(f1.x * alpha, f1.y * alpha);
                            q0[e] = *reinterpret_cast<uint32_t *>(&g0);
                            q1[e] = *reinterpret_cast<uint32_t *>(&g1);
                        }
                        tst16(tS, q0);
                        tst16(tS + 16, q1);
                    }
                    l_sum *= alpha;
                    tile_sum *= alpha;
                }
                const float mc = m_raw == -INFINITY ? 0.f : m_raw * c;
                // scale and row sums on the paired f32x2 pipe (two lanes of work per instruction)
                const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-mc, -mc);
                uint64_t s01 = f2_pack(0.f, 0.f), s23 = s01;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 4) {
                    const uint64_t a01 = f2_fma(f2_pack(sv[cc], sv[cc + 1]), c2, nm2);
                    const uint64_t a23 = f2_fma(f2_pack(sv[cc + 2], sv[cc + 3]), c2, nm2);
                    const float p0 = fast_exp2(f2_lo(a01)), p1 = fast_exp2(f2_hi(a01));
                    const float p2 = fast_exp2(f2_lo(a23)), p3 = fast_exp2(f2_hi(a23));
                    s01 = f2_add(s01, f2_pack(p0, p1));
                    s23 = f2_add(s23, f2_pack(p2, p3));
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(p0, p1);
                    __nv_bfloat162 h1 = __floats2bfloat162_rn(p2, p3);
                    pk[cc / 2] = *reinterpret_cast<uint32_t *>(&h0);
                    pk[cc / 2 + 1] = *reinterpret_cast<uint32_t *>(&h1);
                }
                const uint64_t s4 = f2_add(s01, s23);
                tile_sum += f2_lo(s4) + f2_hi(s4);
                // P of this chunk (keys 64q .. 64q + 63) over S columns already read: 32q .. 32q + 31
                uint32_t (&p0)[16] = *reinterpret_cast<uint32_t(*)[16]>(pk);
                uint32_t (&p1)[16] = *reinterpret_cast<uint32_t(*)[16]>(pk + 16);
                tst16(tS + q * 32, p0);
                tst16(tS + q * 32 + 16, p1);
            }
            l_sum += tile_sum;
            tst_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.p_full[t]);
            // M-tile 0's warpgroup zeroes the V rows past the last visible key of the ragged context
            // tile and of the tree tile before their PVs (P is 0 there, but 0 x NaN would not be).
            // Waiting on V(j)'s phase is safe here: that stage cannot move past tile j before the
            // PV that this warpgroup's P(j) gates.
            if (t == 0 && (jg == jtail || jg == nctx)) {
                if (!warp_wait(&bars.v_full[j % kVStages], (j / kVStages) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                unsigned char *st = sm + kOffV + (j % kVStages) * kTileBytes;
                // a row is 128 contiguous bytes in each half (the swizzle permutes within the row)
                for (int i = kvalid * 8 + rho; i < (jg == nctx ? kTreeKeys : kNkv) * 8; i += 128) {
                    const int rr = i >> 3, c16 = i & 7;
                    *reinterpret_cast<uint4 *>(st + rr * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(st + kHalf + rr * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.v_clean[jg == nctx ? 1 : 0]);
            }
        }
        // epilogue: O / l to global, bf16; with a context split, the unnormalised partial O and the
        // row's (max in base-2 units, sum) for the merge
        if (kSplit && ok && warp_wait(&bars.o_done[t], 0, abort_flag, p.status)) {
            tc_fence_after();
            const size_t pr = pbase + t * 128 + rho;
            float4 *po = reinterpret_cast<float4 *>(p.part_o + pr * 128);
#pragma unroll
            for (int cc = 0; cc < 128; cc += 16) {
                if (cc >= p.HD) break;
                uint32_t o[16];
                tld16(tO + cc, o);
                tld_wait();
                if (valid)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        po[cc / 4 + e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                                     __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
            }
            if (valid) {
                p.part_ml[pr * 2] = m_raw == -INFINITY ? -INFINITY : m_raw * c;
                p.part_ml[pr * 2 + 1] = l_sum;
            }
        } else if (!kSplit && ok && warp_wait(&bars.o_done[t], 0, abort_flag, p.status)) {
            tc_fence_after();
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
            __nv_bfloat16 *orow = p.out + ((((size_t)l * p.B + b) * p.n + node) * p.Hq + g * p.G + gh) * p.HD;
            // 64 columns of O per TMEM round trip (four loads, one wait)
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 64) {
                if (c0 >= p.HD) break;  // d = 64: the upper half of O is the zero padding's
                uint32_t o[64];
                tld16(tO + c0, *reinterpret_cast<uint32_t(*)[16]>(o));
                tld16(tO + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
                tld16(tO + c0 + 32, *reinterpret_cast<uint32_t(*)[16]>(o + 32));
                tld16(tO + c0 + 48, *reinterpret_cast<uint32_t(*)[16]>(o + 48));
                tld_wait();
#pragma unroll
                for (int cc = 0; cc < 64; cc += 16) {
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        __nv_bfloat162 hh = __floats2bfloat162_rn(__uint_as_float(o[cc + 2 * e]) * inv,
                                                                  __uint_as_float(o[cc + 2 * e + 1]) * inv);
                        w[e] = *reinterpret_cast<uint32_t *>(&hh);
                    }
                    if (valid) {
                        reinterpret_cast<uint4 *>(orow + c0 + cc)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        reinterpret_cast<uint4 *>(orow + c0 + cc)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
        }
    }

    // teardown: let every issued TMA copy land before the shared memory is given up
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        // the last copy issued into each stage has landed (already true unless the CTA aborted)
        for (int j = k_issued > kKStages ? k_issued - kKStages : 0; j < k_issued; ++j)
            mbar_wait_bounded(&bars.k_full[j % kKStages], (j / kKStages) & 1);
        for (int j = v_issued > kVStages ? v_issued - kVStages : 0; j < v_issued; ++j)
            mbar_wait_bounded(&bars.v_full[j % kVStages], (j / kVStages) & 1);
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// The merge of a context split: one warp per query row, each lane four of its 128 outputs.  With
// partial (m_s, l_s, O_s) per split (O_s = sum 2^(s c - m_s) v over the split's keys), the row's
// output is sum_s w_s O_s / sum_s w_s l_s, w_s = 2^(m_s - max_s m_s).
__global__ void __launch_bounds__(256) tree_attn_merge_kernel(AttnTcParams p) {
    pdl_wait();
    pdl_launch_next();
    const long wid = (long(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long total = long(p.L) * p.B * p.Hkv * p.rows;
    if (wid >= total) return;
    const int r = int(wid % p.rows);
    const long unit = wid / p.rows;
    const int g = int(unit % p.Hkv), b = int((unit / p.Hkv) % p.B), l = int(unit / (long(p.Hkv) * p.B));
    const int ctx = p.ctx_len[b];
    if (ctx < 0 || ctx > p.S_max) return;  // flagged by the main kernel; the rows stay unwritten
    const int rpt = attn_tc_rows_per_mtile(p.G);
    const int mg = r / (2 * rpt), rin = r % (2 * rpt);
    const int pin = (rin / rpt) * 128 + rin % rpt;  // M-tile and lane of the row in its CTA's partial
    auto prow = [&](int s) { return ((size_t(unit) * p.splits + s) * p.mgroups + mg) * 256 + pin; };
    // lane s < splits: split s's (max, sum), all loaded at once; the weights by warp reduction
    float ms = -INFINITY, ls = 0.f;
    if (lane < p.splits) {
        const float2 v = reinterpret_cast<const float2 *>(p.part_ml)[prow(lane)];
        ms = v.x;
        ls = v.y;
    }
    float M = ms;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w = (M == -INFINITY || ms == -INFINITY) ? 0.f : exp2f(ms - M);
    float lsum = w * ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    // every split's four outputs of this lane, eight loads in flight at a time
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < p.splits; s0 += 8) {
        float4 o[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            o[u] = s0 + u < p.splits ? reinterpret_cast<const float4 *>(p.part_o + prow(s0 + u) * 128)[lane]
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float ws = __shfl_sync(0xffffffffu, w, (s0 + u) & 31);
            acc.x += ws * o[u].x;
            acc.y += ws * o[u].y;
            acc.z += ws * o[u].z;
            acc.w += ws * o[u].w;
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const int node = r / p.G, gh = r % p.G;
    __nv_bfloat16 *orow = p.out + ((((size_t)l * p.B + b) * p.n + node) * p.Hq + g * p.G + gh) * p.HD;
    if (4 * lane >= p.HD) return;  // d = 64: lanes 16 .. 31 hold the zero padding
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2 *>(orow)[lane] =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3-D map over a [outer][mid][hd] bf16 tensor with a {64, box_mid, box_outer} 128B-swizzled box
// (hd = 64: a box at x = 64 lies past the tensor and lands as zeros)
bool make_map(CUtensorMap *map, const void *base, uint64_t hd, uint64_t mid, uint64_t outer, uint32_t box_mid,
              uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {hd, mid, outer};
    cuuint64_t strides[2] = {hd * 2, mid * hd * 2};
    cuuint32_t box[3] = {64, box_mid, box_outer};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over a [rows][heads][hd] bf16 tensor seen as {64 elems, rows, hd / 64 halves, heads}
// (strides out of order) with a {64, box_rows, box_halves, 1} 128B-swizzled box (hd = 64: the
// second half of a two-half box lies past the tensor and lands as zeros).
bool make_kv_map(CUtensorMap *map, const void *base, uint64_t hd, uint64_t heads, uint64_t rows, uint32_t box_rows,
                 uint32_t box_halves) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, rows, hd / 64, heads};
    cuuint64_t strides[3] = {heads * hd * 2, 128, hd * 2};
    cuuint32_t box[4] = {64, box_rows, box_halves, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// True when the tensor-core kernel handles this configuration.
bool tree_attention_tc_supported(int head_dim, int dtype, int G, int S_max) {
    return dtype == EAGLE_DTYPE_BF16 && (head_dim == 128 || head_dim == 64) && G >= 1 && G <= 128 && S_max >= 1 &&
           encode_fn() != nullptr;
}

eagle_status tree_attention_tc_launch(const AttnTcParams &p, const void *q, const void *k_cache, const void *v_cache,
                                      const void *k_tree, const void *v_tree, cudaStream_t stream) {
    CUtensorMap qm, km, vm, ktm, vtm;
    const uint64_t LB = uint64_t(p.L) * p.B;
    const uint64_t hd = uint64_t(p.HD);
    if (!make_map(&qm, q, hd, p.Hq, LB * p.n, p.G, 128 / p.G) ||
        !make_kv_map(&km, k_cache, hd, p.Hkv, LB * p.S_max, kNkv, 2) ||
        !make_kv_map(&vm, v_cache, hd, p.Hkv, LB * p.S_max, kNkv, 2) ||
        !make_kv_map(&ktm, k_tree, hd, p.Hkv, LB * p.n, kNkv, 2) || !make_kv_map(&vtm, v_tree, hd, p.Hkv, LB * p.n, kNkv, 2))
        return EAGLE_ERR_UNSUPPORTED;  // the caller falls back to the mma.sync kernel
    static std::atomic<uint64_t> ready{0};
    const size_t smem = kSmemBytes + 1024;
    if (once_per_device(ready, [&] {
            cudaError_t e =
                cudaFuncSetAttribute(tree_attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(tree_attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
            return e;
        }) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    const long grid = long(p.L) * p.B * p.Hkv * p.mgroups * p.splits;
    const cudaError_t e = p.splits > 1 ? launch_pdl(tree_attn_tc_kernel<true>, dim3(unsigned(grid)), dim3(kThreads), smem,
                                                    stream, 1u, qm, km, vm, ktm, vtm, p)
                                       : launch_pdl(tree_attn_tc_kernel<false>, dim3(unsigned(grid)), dim3(kThreads),
                                                    smem, stream, 1u, qm, km, vm, ktm, vtm, p);
    if (e != cudaSuccess) return EAGLE_ERR_CUDA;
    note_launch();
    if (p.splits > 1) {
        const long warps = long(p.L) * p.B * p.Hkv * p.rows;
        if (launch_pdl(tree_attn_merge_kernel, dim3(unsigned((warps + 7) / 8)), dim3(256), 0, stream, 1u, p) !=
            cudaSuccess)
            return EAGLE_ERR_CUDA;
        note_launch();
    }
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // namespace eagle
