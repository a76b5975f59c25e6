// K2: the K/V projection out[l] = normed[l] x W[l] on the 5th-generation
// tensor cores (tcgen05.mma kind::f16, BF16 in, FP32 accumulate in TMEM).
//
// Page "vllm.models.muse_spark.nvidia.specialized_decode.runtime.draft",
// ContextKV._project: torch.bmm(per_layer [L, T, D], W^T) -> [L, T, 2*H*64].
// The pages leave this GEMM to cuBLAS; this is a hand-written sm_103a
// kernel instead.
//
// Design (one CTA per 128 x BN output tile of one layer and one K split):
//   warp 0     one lane issues TMA tile loads (A: 128 rows x 64 K, B: 64 K x
//              BN) into a STAGES-deep ring of 128-byte-swizzled smem stages;
//   warp 1     allocates BN TMEM columns; one lane issues 4 MMAs of
//              128 x BN x 16 per stage and commits each stage back to the
//              loader, then commits the accumulator to the epilogue;
//   warps 2-5  read the accumulator out of TMEM (warp w owns lanes
//              32*(w%4) ...), round to bf16 (or keep FP32 partials for
//              split-K) and store rows straight to global memory.
// Every wait on an mbarrier is bounded by wall time; on timeout the kernel
// raises a sticky fault bit, skips its remaining work, drains its own copies
// and frees its TMEM.
#include "rc_internal.cuh"
#include "rc_tcgen05.cuh"

#include <algorithm>

namespace rc {

__device__ unsigned int g_project_faults;

namespace {

constexpr int BM = 128;
constexpr int BK = 64;                    // one 128-byte swizzle row of bf16
constexpr int kThreads = 192;
constexpr uint32_t kABytes = BM * BK * 2; // 16 KiB per stage

enum : unsigned { kFaultLoad = 1u, kFaultMma = 2u, kFaultAccum = 4u, kFaultDrain = 8u };

__device__ __forceinline__ bool faulted() {
    return *reinterpret_cast<volatile unsigned int *>(&g_project_faults) != 0u;
}

__device__ __forceinline__ void raise_fault(unsigned bit) { atomicOr(&g_project_faults, bit); }

// Wait for the phase with `parity` to complete; false after the time limit
// or when another CTA of any projection has already raised a fault.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_wait_flag(bar, parity, &g_project_faults);
}

struct GemmArgs {
    int32_t T, N, L;
    int32_t kb_total, kb_per_split, splits;
    uint16_t *out;       // bf16 [L, T, N] when splits == 1
    float *partial;      // FP32 [splits, L, T, N] when splits > 1
    // Pair kernel forming A in shared memory (fused norms): A = z [T, D]
    // scaled per row by row_scale and per column by col_gain [L, D] (or 1)
    const float *row_scale;
    const uint16_t *col_gain;
};

template <int BN>
struct Cfg {
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr uint32_t kBBytes = BN * BK * 2;
    static constexpr uint32_t kStageTx = kABytes + kBBytes;
    static constexpr size_t kSmem = 1024 + (size_t)kStages * (kABytes + kBBytes) + 256;
};

__device__ __forceinline__ uint32_t pack_acc(uint32_t a, uint32_t b) {
    return pack_bf16x2(__uint_as_float(a), __uint_as_float(b));
}

template <int BN, bool kBmn>
__global__ void __launch_bounds__(kThreads, 1)
k2_project(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const GemmArgs g)
{
    using C = Cfg<BN>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + S * kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * (kABytes + C::kBBytes));
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t accum = bar0 + 8u * (2 * S);
    // words[0]: TMEM base address; words[1]: stages the MMA thread consumed
    volatile uint32_t *words = reinterpret_cast<volatile uint32_t *>(bars + 2 * S + 1);

    const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * BM;
    const int l = blockIdx.z / g.splits;
    const int split = blockIdx.z - l * g.splits;
    const int kb0 = split * g.kb_per_split;
    const int nkb = min(g.kb_per_split, g.kb_total - kb0);
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar0 + 8u * s, 1);          // full[s]: the loader's expect_tx
            mbar_init(bar0 + 8u * (S + s), 1);    // empty[s]: the MMA thread's commit
        }
        mbar_init(accum, 1);
        words[1] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32((const void *)words)), "r"(BN) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = words[0];
    if (warp == 0 && lane == 0) {
        // the first stages' weights into L2 while the previous kernel
        // finishes (a hint: the loads below still wait for it)
        for (int i = 0; i < min(nkb, S); ++i) {
            const int kc = (kb0 + i) * BK;
            if (kBmn) {
                for (int c = 0; c < BN / 64; ++c)
                    tma_prefetch_3d(&tmB, n0 + 64 * c, kc, l);
            } else {
                tma_prefetch_3d(&tmB, kc, n0, l);
            }
        }
    }
    pdl_wait();                                   // the previous kernel's writes are visible
    const bool skip = faulted();

    int issued = 0;
    if (warp == 0) {
        if (lane == 0 && !skip) {
            for (int i = 0; i < nkb; ++i) {
                const int s = i % S;
                const uint32_t ph = (uint32_t)(i / S) & 1u;
                if (!mbar_wait(bar0 + 8u * (S + s), ph ^ 1u)) {
                    raise_fault(kFaultLoad);
                    break;
                }
                const uint32_t full = bar0 + 8u * s;
                mbar_expect_tx(full, C::kStageTx);
                const int kc = (kb0 + i) * BK;
                tma_load_3d(sA + s * kABytes, &tmA, kc, m0, l, full);
                if (kBmn) {
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c)
                        tma_load_3d(sB + s * C::kBBytes + c * 8192u, &tmB, n0 + 64 * c, kc, l, full);
                } else {
                    tma_load_3d(sB + s * C::kBBytes, &tmB, kc, n0, l, full);
                }
                issued = i + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int consumed = 0;
            if (!skip) {
                constexpr uint32_t idesc = make_idesc(BM, BN, kBmn);
                for (int i = 0; i < nkb; ++i) {
                    const int s = i % S;
                    const uint32_t ph = (uint32_t)(i / S) & 1u;
                    if (!mbar_wait(bar0 + 8u * s, ph)) {
                        raise_fault(kFaultMma);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = sA + s * kABytes, b = sB + s * C::kBBytes;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // A: K-major, 8-row groups 1024 B apart; +32 B per 16 K.
                        const uint64_t ad = smem_desc_sw128(a + 32u * kk, 16u, 1024u);
                        // B: MN-major: 64-wide N chunks 8 KiB apart, 8-row K
                        // groups 1024 B apart, +2 KiB per 16 K; K-major like A.
                        const uint64_t bd = kBmn ? smem_desc_sw128(b + 2048u * kk, 8192u, 1024u)
                                                 : smem_desc_sw128(b + 32u * kk, 16u, 1024u);
                        mma_bf16(tmem, ad, bd, idesc, (i | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(bar0 + 8u * (S + s));   // frees the stage when these MMAs finish
                    consumed = i + 1;
                }
            }
            words[1] = (uint32_t)consumed;
            mma_commit(accum);                        // all MMAs issued above are done
        }
        __syncwarp();
    } else {
        const int q = warp & 3;                       // TMEM lane quadrant of this warp
        bool ok = !skip && mbar_wait(accum, 0u);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok && !skip && lane == 0)
            raise_fault(kFaultAccum);
        if (ok) {
            tc_fence_after();
            const int row = m0 + 32 * q + lane;
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tbase + 32u * c, r);
                if (row < g.T) {
                    if (g.splits == 1) {
                        uint4 *o = reinterpret_cast<uint4 *>(
                            g.out + ((int64_t)l * g.T + row) * g.N + n0 + 32 * c);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            o[j] = make_uint4(pack_acc(r[8 * j], r[8 * j + 1]),
                                              pack_acc(r[8 * j + 2], r[8 * j + 3]),
                                              pack_acc(r[8 * j + 4], r[8 * j + 5]),
                                              pack_acc(r[8 * j + 6], r[8 * j + 7]));
                    } else {
                        float4 *o = reinterpret_cast<float4 *>(
                            g.partial + (((int64_t)split * g.L + l) * g.T + row) * g.N + n0 + 32 * c);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            o[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                               __uint_as_float(r[4 * j + 2]),
                                               __uint_as_float(r[4 * j + 3]));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        // Loads issued but never consumed exist only after a fault: wait for
        // them to land before the CTA's shared memory goes away.
        for (int i = (int)words[1]; i < issued; ++i)
            if (!mbar_wait_own(bar0 + 8u * (i % S), (uint32_t)(i / S) & 1u)) {
                raise_fault(kFaultDrain);
                break;
            }
    }
    if (warp == 1) {
        if (lane == 0 && !mbar_wait_own(accum, 0u))
            raise_fault(kFaultDrain);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BN)
                     : "memory");
    }
}

// out = bf16(sum over splits of the FP32 partials), added in split order.
__global__ void __launch_bounds__(256)
k2_splitk_reduce(const float *__restrict__ partial, uint16_t *__restrict__ out, int64_t count,
                 int splits)
{
    const int64_t n8 = count / 8;
    pdl_trigger();
    pdl_wait();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 *p = reinterpret_cast<const float4 *>(partial) + 2 * i;
        float4 a = __ldcs(p), b = __ldcs(p + 1);
        for (int s = 1; s < splits; ++s) {
            const float4 *q = p + (int64_t)s * (count / 4);
            const float4 c = __ldcs(q), d = __ldcs(q + 1);
            a.x = __fadd_rn(a.x, c.x); a.y = __fadd_rn(a.y, c.y);
            a.z = __fadd_rn(a.z, c.z); a.w = __fadd_rn(a.w, c.w);
            b.x = __fadd_rn(b.x, d.x); b.y = __fadd_rn(b.y, d.y);
            b.z = __fadd_rn(b.z, d.z); b.w = __fadd_rn(b.w, d.w);
        }
        reinterpret_cast<uint4 *>(out)[i] =
            make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                       pack_bf16x2(b.z, b.w));
    }
}

// ------------------------------------------------------------- CTA pairs
//
// k2_project_pair: the same tile pipeline on a pair of CTAs (a cluster of 2
// on neighbouring SMs) issuing tcgen05.mma.cta_group::2 with M = 256, N = 256.
// CTA r of the pair stages A rows m0 + 128 r ... and B columns n0 + 128 r ...
// (half of B each), so one 256 x 256 x 64 step moves 32 KiB into each SM
// instead of the 48 KiB a single-CTA 128 x 256 tile needs, and 6 stages fit
// where 4 did.  The leader (rank 0) waits for both CTAs' bytes on its own
// barriers and issues the MMAs; commits arrive on both CTAs' barriers.  Each
// CTA's TMEM holds the accumulator of its own 128 rows.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
    return d;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// TMA load into this CTA's smem whose bytes are counted on `bar`, a barrier
// of the pair's leader (a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, int c0,
                                                 int c1, int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` (same offset) in both CTAs of the pair once the MMAs
// issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"((uint16_t)0x3) : "memory");
}

// ------------------------------------------------- fused store epilogue
//
// With the projection and the store fused, an epilogue thread holds its row's
// 256 accumulators = 4 heads of K or of V.  It rounds them to bf16 (the
// projection), and for a key head computes the K-norm from those bf16 values
// with the sum folded exactly as the store kernel's lane butterfly does it
// (seen from lane 0: pairs (j, j+16), then +8, +4, +2, +1 partners; even
// and odd squares separately, then even + odd), so the stored key is the
// same bits the unfused store would write.

// One head of the warp's 32 rows (w: this lane's row, 32 packed bf16 pairs)
// leaves for memory through the warp's staging rows in shared memory (32
// rows 144 bytes apart: conflict-free both ways), so that each store
// instruction writes four whole 128-byte rows instead of 32 scattered 16-byte
// pieces.  dst: this lane's destination row (64 bf16), or NULL; every lane
// takes part.
__device__ __forceinline__ void store_head_rows(uint32_t stage, int lane, const uint32_t (&w)[32],
                                                uint16_t *dst) {
    const uint32_t own = stage + (uint32_t)lane * 144u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        st_shared_v4(own + 16u * j, make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]));
    __syncwarp();
    const int piece = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane >> 3) + 4 * i;
        uint16_t *d = reinterpret_cast<uint16_t *>(
            __shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(dst), r));
        const uint4 v = ld_shared_v4(stage + (uint32_t)r * 144u + 16u * piece);
        if (d != nullptr)
            reinterpret_cast<uint4 *>(d)[piece] = v;
    }
    __syncwarp();                                      // reads done before the next head's writes
}

// The tile's store for one row (all 32 lanes call it: TMEM loads and the
// staged stores are warp-collective).  tbase: this warp's TMEM lanes, column
// 0 of the tile; stage: the warp's staging rows (32 x 144 bytes).
// kPreload: the table row is read once per tile (in registers), else once
// per key head (for kernels that cannot spare the registers).
template <bool kPreload>
__device__ __forceinline__ void fused_store_tile(const FusedStore &fs, const GemmArgs &g,
                                                 uint32_t tbase, int l, int row, int n0,
                                                 uint32_t stage, int lane) {
    const bool live = row < g.T;
    const bool rope = fs.cos_sin != nullptr;
    const int H = fs.H;
    const int N = g.N;
    bool store = false;
    int64_t slot = 0, pos = 0;
    if (live && row < fs.rows[l] && fs.slots[l] != nullptr) {
        slot = __ldg(fs.slots[l] + row);
        if (slot >= 0) {
            if (rope)
                pos = __ldg(fs.positions + row);
            if (slot >= fs.capacity || (rope && (pos < 0 || pos >= fs.max_position))) {
                if (n0 == 0 && fs.err != nullptr)        // counted once per (row, layer)
                    atomicAdd(fs.err, 1);
            } else {
                store = true;
            }
        }
    }
    uint16_t *dst_row = nullptr;                       // this row's cache row, head 0
    if (store) {
        const uint32_t bs = (uint32_t)fs.block_size;
        const uint32_t blk = (uint32_t)slot / bs;
        const uint32_t page = (uint32_t)slot - blk * bs;
        dst_row = fs.caches[l] + (((int64_t)blk * H) * bs + page) * (2 * kHeadDim);
    }
    // the row's cos | sin table row, fetched once for the tile's key heads
    uint4 cq[4], sq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        cq[q] = sq[q] = make_uint4(0, 0, 0, 0);
    const uint4 *cs = rope && store ? reinterpret_cast<const uint4 *>(fs.cos_sin + pos * kHeadDim) : nullptr;
    if (kPreload && cs != nullptr && (n0 >> 6) < H) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            cq[q] = __ldg(cs + q);                     // cos of pairs 8q .. 8q+7
            sq[q] = __ldg(cs + 4 + q);                 // sin of the same pairs
        }
    }
#pragma unroll 1
    for (int hh = 0; hh < 4; ++hh) {
        uint32_t r[64];
        tmem_ld32(tbase + 64u * hh, *reinterpret_cast<uint32_t (*)[32]>(r));
        tmem_ld32(tbase + 64u * hh + 32u, *reinterpret_cast<uint32_t (*)[32]>(r + 32));
        uint32_t kp[32];                               // the projection, bf16 pairs
#pragma unroll
        for (int j = 0; j < 32; ++j)
            kp[j] = pack_acc(r[2 * j], r[2 * j + 1]);
        if (fs.kv_out != nullptr)
            store_head_rows(stage, lane, kp,
                            live ? fs.kv_out + ((int64_t)l * g.T + row) * N + n0 + 64 * hh : nullptr);
        const int gidx = (n0 >> 6) + hh;               // head index within [K heads | V heads]
        const bool is_k = gidx < H;                    // the same for the whole warp
        const int h = is_k ? gidx : gidx - H;
        uint16_t *dst = store ? dst_row + (int64_t)h * fs.block_size * (2 * kHeadDim) + (is_k ? 0 : kHeadDim)
                              : nullptr;
        if (is_k) {
            // the K-norm's even and odd square sums in the store kernel's
            // fold order, then the bf16 key and its rotation per pair
            float even, odd;
            fold32_squares2(kp, even, odd);
            const float rr = inv_rms(__fadd_rn(even, odd), 0x1p-6f, fs.eps);
#pragma unroll
            for (int q = 0; q < 4; ++q) {              // 8 pairs at a time
                if (!kPreload && cs != nullptr) {
                    cq[q] = __ldg(cs + q);
                    sq[q] = __ldg(cs + 4 + q);
                }
                const uint32_t cw[4] = {cq[q].x, cq[q].y, cq[q].z, cq[q].w};
                const uint32_t sw[4] = {sq[q].x, sq[q].y, sq[q].z, sq[q].w};
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int j = 8 * q + t;
                    const float c = (t & 1) ? bf16_hi(cw[t >> 1]) : bf16_lo(cw[t >> 1]);
                    const float sn = (t & 1) ? bf16_hi(sw[t >> 1]) : bf16_lo(sw[t >> 1]);
                    kp[j] = rope ? norm_rope_pair<true>(kp[j], rr, c, sn)
                                 : norm_rope_pair<false>(kp[j], rr, c, sn);
                }
            }
        }
        store_head_rows(stage, lane, kp, dst);         // K' (or V, a bit copy of the projection)
    }
}

// Staging rows of one epilogue warp: 32 rows of 144 bytes (FP32) or 80
// bytes (bf16), placed in the first pipeline stage.
constexpr uint32_t kStageRowsBytes = 32u * 144u;

struct PairCfg {
    static constexpr int kStages = 6;
    static constexpr uint32_t kBHalf = 128 * BK * 2;            // 16 KiB of B per CTA
    static constexpr uint32_t kStageBytes = kABytes + kBHalf;    // 32 KiB per CTA
    static constexpr uint32_t kPairTx = 2 * kStageBytes;         // counted on the leader
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + 512;
    static_assert((5 * kStages + 1) * 8 + 5 * 4 <= 512, "barriers and words fit the tail");
    static_assert(4 * kStageRowsBytes <= (uint32_t)kStages * kABytes, "staging rows fit the A stages");
};

__device__ __forceinline__ void unpack8f(const uint4 &q, float *f) {
    f[0] = bf16_lo(q.x); f[1] = bf16_hi(q.x);
    f[2] = bf16_lo(q.y); f[3] = bf16_hi(q.y);
    f[4] = bf16_lo(q.z); f[5] = bf16_hi(q.z);
    f[6] = bf16_lo(q.w); f[7] = bf16_hi(q.w);
}

// One 8-value chunk of a layer's normed row from the hidden-norm output z:
// bf16((z * rs) * gm[e]) per value (gm == nullptr: bf16(z * rs)), the
// operations and roundings of the norms kernel's layer step.
__device__ __forceinline__ uint4 form_chunk(const uint4 &v, float rs, const float *gm) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float lo = bf16_lo(w[k]), hi = bf16_hi(w[k]);
        mul2_rn(lo, hi, rs, rs);
        if (gm != nullptr)
            mul2_rn(lo, hi, gm[2 * k], gm[2 * k + 1]);
        o[k] = pack_bf16x2(lo, hi);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// kTransform: the A tile is formed in shared memory from the hidden-norm
// output z (TMA-loaded): A = bf16((z * row_scale) * col_gain_l), the same
// operations and roundings as the norms kernel's layer step, so the operand
// is bit-identical to the normed rows that kernel would have written.  The
// 4 epilogue warps do it in place (128-byte swizzled rows: logical 16-byte
// chunk c of row r sits at chunk c ^ (r % 8)) before the epilogue.
// Threads of the pair kernel: producer warp, MMA warp, 4 epilogue warps
// (with kTransform: kFormGroups groups of 4 forming warps taking stages in
// turn, so several stages are formed at once; warps 2-5 also run the
// epilogue).
constexpr int kFormGroups = 3;
template <bool kTransform>
constexpr int pair_threads() { return kTransform ? 64 + 128 * kFormGroups : kThreads; }

template <bool kBmn, bool kFused, bool kTransform>
__global__ void __launch_bounds__(pair_threads<kTransform>(), 1)
k2_project_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs g, const __grid_constant__ FusedStore fs)
{
    using C = PairCfg;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + S * kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * C::kStageBytes);
    // full[s] (leader: B, and A unless kTransform), empty[s], aload[s]
    // (kTransform: this CTA's A), ready[s] (kTransform: this CTA's A is
    // formed), peer[s] (kTransform, leader: the peer's A is formed), accum
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t empty0 = bar0 + 8u * S, aload0 = bar0 + 16u * S, ready0 = bar0 + 24u * S;
    const uint32_t peer0 = bar0 + 32u * S;
    const uint32_t accum = bar0 + 40u * S;
    // words[0]: TMEM base; [1]: stages the leader's MMA thread consumed;
    // [2]: skip flag (written by the leader into both CTAs); [3]: stages the
    // peer's loader issued (written by the peer into the leader)
    volatile uint32_t *words = reinterpret_cast<volatile uint32_t *>(bars + 5 * S + 1);
    const uint32_t words_addr = smem_u32((const void *)words);

    const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int n0 = (blockIdx.x >> 1) * 256;        // the pair's 256 output columns
    const int m0 = blockIdx.y * 256 + 128 * (int)rank;   // this CTA's 128 rows
    const int nb = n0 + 128 * (int)rank;           // this CTA's half of B
    const int l = blockIdx.z / g.splits;
    const int split = blockIdx.z - l * g.splits;
    const int kb0 = split * g.kb_per_split;
    const int nkb = min(g.kb_per_split, g.kb_total - kb0);
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
            mbar_init(aload0 + 8u * s, 1);
            mbar_init(ready0 + 8u * s, 4);         // the 4 forming warps of the stage's group
            mbar_init(peer0 + 8u * s, 1);          // forwarded by the peer's warp 1
        }
        mbar_init(accum, 1);
        words[1] = 0u;
        words[3] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (leader) {
            // One skip decision for the pair, written into both CTAs.  Read
            // before pdl_wait: a fault raised by a projection still finishing
            // just before this one can be missed, and this one then runs.
            const uint32_t skip = faulted() ? 1u : 0u;
            words[2] = skip;
            st_cluster_u32(map_to_rank(words_addr + 8u, 1), skip);
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(words_addr), "r"(256) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();                               // barriers, skip flag and TMEM pair-wide
    tc_fence_after();
    const uint32_t tmem = words[0];
    const bool skip = words[2] != 0u;
    if (warp == 0 && lane == 0) {
        // the first stages' weights into L2 while the previous kernel
        // finishes (a hint: the loads below still wait for it)
        for (int i = 0; i < min(nkb, S); ++i) {
            const int kc = (kb0 + i) * BK;
            if (kBmn) {
                tma_prefetch_3d(&tmB, nb, kc, l);
                tma_prefetch_3d(&tmB, nb + 64, kc, l);
            } else {
                tma_prefetch_3d(&tmB, kc, nb, l);
            }
        }
    }
    pdl_wait();                                   // the previous kernel's writes are visible

    int issued = 0;
    if (warp == 0) {
        if (lane == 0 && !skip) {
            for (int i = 0; i < nkb; ++i) {
                const int s = i % S;
                const uint32_t ph = (uint32_t)(i / S) & 1u;
                if (!mbar_wait(empty0 + 8u * s, ph ^ 1u)) {
                    raise_fault(kFaultLoad);
                    break;
                }
                const uint32_t full = map_to_rank(bar0 + 8u * s, 0);
                if (leader)
                    mbar_expect_tx(bar0 + 8u * s, kTransform ? 2u * C::kBHalf : C::kPairTx);
                const int kc = (kb0 + i) * BK;
                if (kTransform) {
                    mbar_expect_tx(aload0 + 8u * s, kABytes);
                    tma_load_3d(sA + s * kABytes, &tmA, kc, m0, 0, aload0 + 8u * s);
                } else {
                    tma_load_3d_pair(sA + s * kABytes, &tmA, kc, m0, l, full);
                }
                if (kBmn) {
                    tma_load_3d_pair(sB + s * C::kBHalf, &tmB, nb, kc, l, full);
                    tma_load_3d_pair(sB + s * C::kBHalf + 8192u, &tmB, nb + 64, kc, l, full);
                } else {
                    tma_load_3d_pair(sB + s * C::kBHalf, &tmB, kc, nb, l, full);
                }
                issued = i + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int consumed = 0;
            if (!skip) {
                constexpr uint32_t idesc = make_idesc(256, 256, kBmn);
                for (int i = 0; i < nkb; ++i) {
                    const int s = i % S;
                    const uint32_t ph = (uint32_t)(i / S) & 1u;
                    if (!mbar_wait(bar0 + 8u * s, ph) ||
                        (kTransform && (!mbar_wait(ready0 + 8u * s, ph) ||
                                        !mbar_wait(peer0 + 8u * s, ph)))) {
                        raise_fault(kFaultMma);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = sA + s * kABytes, b = sB + s * C::kBHalf;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(a + 32u * kk, 16u, 1024u);
                        const uint64_t bd = kBmn ? smem_desc_sw128(b + 2048u * kk, 8192u, 1024u)
                                                 : smem_desc_sw128(b + 32u * kk, 16u, 1024u);
                        mma_bf16_pair(tmem, ad, bd, idesc, (i | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit_pair(empty0 + 8u * s);
                    consumed = i + 1;
                }
            }
            words[1] = (uint32_t)consumed;
            mma_commit_pair(accum);
        } else if (kTransform && lane == 0 && !skip) {
            // The peer's idle MMA thread forwards "A formed" to the leader, so
            // the forming warps never pay for a cluster-scope release.
            const uint32_t peer_lead = map_to_rank(peer0, 0);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % S;
                if (!mbar_wait(ready0 + 8u * s, (uint32_t)(i / S) & 1u)) {
                    raise_fault(kFaultMma);
                    break;
                }
                mbar_arrive_cluster(peer_lead + 8u * s);
            }
        }
        __syncwarp();
    } else {
        const int q = warp & 3;
        if (kTransform && !skip) {
            // Form this CTA's A tiles: group grp (warps 2 + 4 grp ...) forms
            // the stages i with i % kFormGroups == grp; thread t of a group
            // takes logical chunk c = t % 8 (8 columns) of rows t / 8 + 16 j.
            const int grp = ((int)threadIdx.x - 64) >> 7;
            const int t = ((int)threadIdx.x - 64) & 127;
            const int c = t & 7, r0 = t >> 3;
            float rs[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int row = m0 + r0 + 16 * j;
                rs[j] = row < g.T ? __ldg(g.row_scale + row) : 0.0f;
            }
            const uint16_t *gain =
                g.col_gain ? g.col_gain + (int64_t)l * (g.kb_total * BK) + 8 * c : nullptr;
            // the gains of the group's next stage are fetched while the
            // current one is formed, so no stage waits for them
            uint4 g_next = make_uint4(0, 0, 0, 0);
            if (gain && grp < nkb)
                g_next = __ldg(reinterpret_cast<const uint4 *>(gain + (kb0 + grp) * BK));
            for (int i = grp; i < nkb; i += kFormGroups) {
                const int s = i % S;
                const uint32_t ph = (uint32_t)(i / S) & 1u;
                float gm[8];
                if (gain) {
                    unpack8f(g_next, gm);
                    if (i + kFormGroups < nkb)
                        g_next = __ldg(reinterpret_cast<const uint4 *>(gain + (kb0 + i + kFormGroups) * BK));
                }
                if (!mbar_wait(aload0 + 8u * s, ph)) {
                    raise_fault(kFaultLoad);
                    break;
                }
                // all 8 rows' chunks in flight, then formed, then written
                // back; rows r0 + 16 j share r % 8, so their swizzled chunks
                // sit 2048 bytes apart from one base
                const uint32_t base = sA + s * kABytes + r0 * 128 + ((c ^ (r0 & 7)) << 4);
                uint4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v[j] = ld_shared_v4(base + 2048u * j);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v[j] = form_chunk(v[j], rs[j], gain ? gm : nullptr);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(base + 2048u * j, v[j]);
                // generic-proxy writes, then visible to the tensor core
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_local(ready0 + 8u * s);
            }
        }
        bool ok = warp < 6 && !skip && mbar_wait(accum, 0u);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok && !skip && warp < 6 && lane == 0)
            raise_fault(kFaultAccum);
        if (ok && kFused && g.splits == 1) {
            tc_fence_after();
            fused_store_tile<!kTransform>(fs, g, tmem + ((uint32_t)(32 * q) << 16), l, m0 + 32 * q + lane, n0,
                             sA + (uint32_t)q * kStageRowsBytes, lane);
        } else if (ok) {
            // Each thread holds one row's 32 accumulators per TMEM load; they
            // pass through this warp's staging rows in shared memory (the
            // pipeline stages are idle once the accumulator is complete) so
            // that every global store instruction writes whole 128-byte (FP32)
            // or 64-byte (bf16) row segments instead of 32 scattered pieces.
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16);
            const uint32_t stage = sA + (uint32_t)q * kStageRowsBytes;
            const int row0 = m0 + 32 * q;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t r[32];
                tmem_ld32(tbase + 32u * c, r);
                if (g.splits == 1) {
                    // bf16: 64 bytes per row, rows 80 bytes apart (conflict-free)
                    const uint32_t w = stage + (uint32_t)lane * 80u;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        st_shared_v4(w + 16u * j, make_uint4(pack_acc(r[8 * j], r[8 * j + 1]),
                                                             pack_acc(r[8 * j + 2], r[8 * j + 3]),
                                                             pack_acc(r[8 * j + 4], r[8 * j + 5]),
                                                             pack_acc(r[8 * j + 6], r[8 * j + 7])));
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = (lane >> 2) + 8 * i, piece = lane & 3;
                        const uint4 v = ld_shared_v4(stage + (uint32_t)rr * 80u + 16u * piece);
                        const int row = row0 + rr;
                        if (row < g.T)
                            *reinterpret_cast<uint4 *>(g.out + ((int64_t)l * g.T + row) * g.N + n0 +
                                                       32 * c + 8 * piece) = v;
                    }
                } else {
                    // FP32 partials: 128 bytes per row, rows 144 bytes apart
                    const uint32_t w = stage + (uint32_t)lane * 144u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(w + 16u * j, make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2],
                                                             r[4 * j + 3]));
                    __syncwarp();
                    float *base = g.partial + ((int64_t)split * g.L + l) * g.T * g.N + n0 + 32 * c;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = (lane >> 3) + 4 * i, piece = lane & 7;
                        const uint4 v = ld_shared_v4(stage + (uint32_t)rr * 144u + 16u * piece);
                        const int row = row0 + rr;
                        if (row < g.T)
                            *reinterpret_cast<uint4 *>(base + (int64_t)row * g.N + 4 * piece) = v;
                    }
                }
                __syncwarp();                        // reads done before the next chunk's writes
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (!leader && warp == 0 && lane == 0)
        st_cluster_u32(map_to_rank(words_addr + 12u, 0), (uint32_t)issued);
    cluster_sync();
    if (warp == 0 && lane == 0) {
        if (leader) {
            // Both CTAs' B (and A) loads land on the leader's barriers: after
            // a fault, wait for every stage either CTA issued before anyone
            // frees smem.
            const int last = max(issued, (int)words[3]);
            for (int i = (int)words[1]; i < last; ++i)
                if (!mbar_wait_own(bar0 + 8u * (i % S), (uint32_t)(i / S) & 1u)) {
                    raise_fault(kFaultDrain);
                    break;
                }
        }
        if (kTransform)                               // this CTA's own A loads
            for (int i = max(0, issued - S); i < issued; ++i)
                if (!mbar_wait_own(aload0 + 8u * (i % S), (uint32_t)(i / S) & 1u)) {
                    raise_fault(kFaultDrain);
                    break;
                }
    }
    if (leader && warp == 1 && lane == 0 && !mbar_wait_own(accum, 0u))
        raise_fault(kFaultDrain);
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256)
                     : "memory");
    }
}

// ------------------------------------------------- persistent CTA pairs
//
// k2_project_pair_persistent: the pair kernel for plans that do not split
// K, with one CTA pair per two SMs taking output tiles t, t + P, t + 2P, ...
// (P pairs; consecutive tiles share A rows and W columns in L2).  The TMA
// ring runs on across tiles, and TMEM holds two 256-column accumulators:
// while the epilogue warps of both CTAs store tile j from one, the MMA
// thread already accumulates tile j + 1 into the other, so the epilogue and
// the per-CTA set-up and pipeline fill no longer sit between mainloops.
// The epilogue (bf16 rows or the fused store) is the pair kernel's.

struct PersistCfg {
    static constexpr int kStages = PairCfg::kStages;
    static constexpr uint32_t kStageBytes = PairCfg::kStageBytes;
    // staging rows of the 4 epilogue warps: 32 rows of 144 bytes each (the
    // fused store's 128-byte head rows; the bf16 rows use 80 bytes of each)
    static constexpr uint32_t kStagingBytes = 4u * kStageRowsBytes;
    static constexpr uint32_t kTailBytes = 1024;   // barriers and words
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kStagingBytes + kTailBytes;
    static_assert((5 * kStages + 13) * 8 + 8 * 4 <= kTailBytes, "barriers and words fit the tail");
};

// Arrive on a barrier of any CTA of the cluster, releasing at cluster scope.
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Dynamic tile order of the persistent kernel.  Each pair's first tile is
// pair_id; after it, the leader's loader of a pair takes the next output
// tile from a counter in global memory when it starts loading it, so tiles
// that share A rows (consecutive indices) start within a fraction of a tile
// time of each other on whichever pairs are free, and their A reads meet in
// L2.  With a fixed assignment over many rounds, the pairs that share A
// drift apart until they read it from DRAM again (2.5 times the A bytes
// measured at 54 rounds).  The call zeroes the counter before the launch.
constexpr int kMaxDynTiles = 1 << 30;

// Bounded wait on a barrier that other CTAs of the cluster arrive on.// Bounded wait on a barrier that other CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok)
            return true;
        if ((it & 255u) == 255u && (faulted() || globaltimer() - t0 > kWaitNs))
            return false;
    }
}

// This warp's 32 rows of a tile as bf16, through the warp's staging rows:
// 64 bytes per row, rows 80 bytes apart (conflict-free), so each global
// store instruction writes whole 64-byte row segments.
__device__ __forceinline__ void write_bf16_rows(const GemmArgs &g, uint32_t tbase, uint32_t stage,
                                                int row0, int l, int n0, int lane) {
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        tmem_ld32(tbase + 32u * c, r);
        const uint32_t w = stage + (uint32_t)lane * 80u;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            st_shared_v4(w + 16u * j, make_uint4(pack_acc(r[8 * j], r[8 * j + 1]),
                                                 pack_acc(r[8 * j + 2], r[8 * j + 3]),
                                                 pack_acc(r[8 * j + 4], r[8 * j + 5]),
                                                 pack_acc(r[8 * j + 6], r[8 * j + 7])));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = (lane >> 2) + 8 * i, piece = lane & 3;
            const uint4 v = ld_shared_v4(stage + (uint32_t)rr * 80u + 16u * piece);
            const int row = row0 + rr;
            if (row < g.T)
                *reinterpret_cast<uint4 *>(g.out + ((int64_t)l * g.T + row) * g.N + n0 + 32 * c +
                                           8 * piece) = v;
        }
        __syncwarp();                                  // reads done before the next chunk's writes
    }
}

// Slots of the ring through which the leader's loader hands out dynamically
// taken tiles (to the peer's loader, the MMA thread and both CTAs' epilogue
// warps), and the readers that release each slot.
constexpr int kTileSlots = 4;
constexpr int kPersistFormGroups = 2;                       // groups taking stages in turn
constexpr int kFormWarpsPerGroup = 4;
constexpr int kFormRows = 32 / kFormWarpsPerGroup;          // rows of a stage per thread
// leader MMA + epilogue, peer loader + epilogue; with forming warps also the
// peer's forwarding thread and both CTAs' forming warps
__host__ __device__ constexpr int tile_readers(bool form) {
    return 1 + 4 + 1 + 4 + (form ? 1 + 2 * kFormWarpsPerGroup * kPersistFormGroups : 0);
}

// Threads of the persistent kernel: loader warp, MMA warp, 4 epilogue warps,
// and with the forming flag kPersistFormGroups groups of 4 forming warps.
__host__ __device__ constexpr int persist_threads(bool form) {
    return kThreads + (form ? 32 * kFormWarpsPerGroup * kPersistFormGroups : 0);
}

// kForm: A is formed in shared memory from the hidden-norm rows z (TMA
// loads of z [T, D] into the A stage, then bf16((z * row_scale) * col_gain_l)
// written in place by the forming warps, as the norms kernel's layer step
// computes it), for the whole chain; kForm implies the fused store.
//
// Register bound without forming: two CTAs per SM (168).  One CTA per SM
// runs (shared memory), and the registers it leaves free hold two 8-warp
// norms CTAs that another stream may run beside it (the end-to-end row
// ranges).
template <bool kBmn, bool kFused, bool kForm>
__global__ void __launch_bounds__(persist_threads(kForm), kForm ? 1 : 2)
k2_project_pair_persistent(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const GemmArgs g,
                           const __grid_constant__ FusedStore fs, int n_pairs, int m_pairs,
                           int tile_limit, unsigned int *tile_ctr)
{
    using C = PersistCfg;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + S * kABytes;
    const uint32_t sStage = sA + S * C::kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * C::kStageBytes + C::kStagingBytes);
    // full[s] (leader: B, and A unless kForm), empty[s], afull[2]
    // (accumulator b complete), aempty[2] (leader: both CTAs' epilogues are
    // done with accumulator b), done, tfull[4] (tile slot written), tempty[4]
    // (leader: slot read by all); with kForm aload[s] (this CTA's z rows
    // landed), ready[s] (this CTA's A formed), peer[s] (leader: the peer's A
    // formed, forwarded by the peer's warp 1)
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t empty0 = bar0 + 8u * S, afull0 = bar0 + 16u * S, aempty0 = afull0 + 16u;
    const uint32_t done = aempty0 + 16u;
    const uint32_t tfull0 = done + 8u, tempty0 = tfull0 + 8u * kTileSlots;
    const uint32_t aload0 = tempty0 + 8u * kTileSlots, ready0 = aload0 + 8u * S, peer0 = ready0 + 8u * S;
    // words[0]: TMEM base; [1]: stages the leader's MMA thread consumed;
    // [2]: skip flag (written by the leader into both CTAs); [3]: stages the
    // peer's loader issued (written by the peer into the leader); [4..7]:
    // the tile slots (written by the leader's loader into both CTAs)
    volatile uint32_t *words = reinterpret_cast<volatile uint32_t *>(bars + 5 * S + 13);
    const uint32_t words_addr = smem_u32((const void *)words);

    const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair_id = (int)(blockIdx.x >> 1), num_pairs = (int)(gridDim.x >> 1);
    // the first tile_limit tiles (the rest, if any, are another launch's)
    const int num_tiles = min(g.L * m_pairs * n_pairs, tile_limit);
    const int nkb = g.kb_total;
    const bool dyn = tile_ctr != nullptr;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(afull0 + 8u * b, 1);
            mbar_init(aempty0 + 8u * b, 8);        // 4 epilogue warps in each CTA of the pair
        }
        mbar_init(done, 1);
        for (int i = 0; i < kTileSlots; ++i) {
            mbar_init(tfull0 + 8u * i, 1);         // the leader's loader
            mbar_init(tempty0 + 8u * i, tile_readers(kForm));
        }
        if (kForm) {
            for (int s = 0; s < S; ++s) {
                mbar_init(aload0 + 8u * s, 1);     // this CTA's loader (expect_tx)
                mbar_init(ready0 + 8u * s, kFormWarpsPerGroup);   // the forming warps of the stage's group
                mbar_init(peer0 + 8u * s, 1);      // forwarded by the peer's warp 1
            }
        }
        words[1] = 0u;
        words[3] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (leader) {
            const uint32_t skip = faulted() ? 1u : 0u;
            words[2] = skip;
            st_cluster_u32(map_to_rank(words_addr + 8u, 1), skip);
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(words_addr), "r"(512) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();                               // barriers, skip flag and TMEM pair-wide
    tc_fence_after();
    const uint32_t tmem = words[0];
    const bool skip = words[2] != 0u;
    if (warp == 0 && lane == 0 && pair_id < num_tiles) {
        // the first tile's first stages of weights into L2 while the
        // previous kernel finishes (a hint: the loads below still wait)
        const int np = pair_id % n_pairs, l = pair_id / n_pairs / m_pairs;
        const int nb = np * 256 + 128 * (int)rank;
        for (int i = 0; i < min(nkb, S); ++i) {
            if (kBmn) {
                tma_prefetch_3d(&tmB, nb, i * BK, l);
                tma_prefetch_3d(&tmB, nb + 64, i * BK, l);
            } else {
                tma_prefetch_3d(&tmB, i * BK, nb, l);
            }
        }
    }
    pdl_wait();                                   // the previous kernel's writes are visible

    // Tile j of this pair: with a fixed order pair_id + j * num_pairs; with
    // dynamic tiles the first one is pair_id and for j >= 1 the leader's
    // loader takes a ticket (publish = true) and every other role reads the
    // tile from slot (j - 1) % 4 and releases the slot.  -1: no more tiles,
    // or a wait that gave up (fault raised).
    const uint32_t tiles_addr = words_addr + 16u;
    const uint32_t lead_tempty0 = map_to_rank(tempty0, 0);
    auto tile_of = [&](int j, bool publish, bool warp_wide) -> int {
        if (!dyn || j == 0) {
            // the fixed sequence; with dynamic tiles the first round as well,
            // so that the pairs do not all take their first ticket at once
            const int t = pair_id + j * num_pairs;
            return t < num_tiles ? t : -1;
        }
        const int slot = (j - 1) % kTileSlots;       // ring use j - 1 (round 0 needs none)
        const uint32_t ph = (uint32_t)((j - 1) / kTileSlots) & 1u;
        if (publish) {
            if (!mbar_wait_cluster(tempty0 + 8u * slot, ph ^ 1u)) {
                raise_fault(kFaultLoad);
                return -1;
            }
            // tickets count the tiles after round 0
            const unsigned int ticket = atomicAdd(tile_ctr, 1u);
            const int t = ticket < (unsigned int)(num_tiles - num_pairs) ? (int)ticket + num_pairs : -1;
            words[4 + slot] = (uint32_t)t;
            st_cluster_u32(map_to_rank(tiles_addr + 4u * slot, 1), (uint32_t)t);
            mbar_arrive_local(tfull0 + 8u * slot);
            mbar_arrive_release_cluster(map_to_rank(tfull0 + 8u * slot, 1));
            return t;
        }
        // one thread waits, reads the slot and releases it (a warp gets the
        // index from its lane 0)
        int t = -1;
        if (!warp_wide || lane == 0) {
            if (mbar_wait_cluster(tfull0 + 8u * slot, ph)) {
                t = (int)words[4 + slot];
                if (leader)
                    mbar_arrive_local(tempty0 + 8u * slot);
                else
                    mbar_arrive_release_cluster(lead_tempty0 + 8u * slot);
            } else {
                raise_fault(kFaultAccum);
            }
        }
        if (warp_wide)
            t = __shfl_sync(0xFFFFFFFFu, t, 0);
        return t;
    };

    int issued = 0;
    if (warp == 0) {
        if (lane == 0 && !skip) {
            int it = 0;
            bool ok = true;
            for (int j = 0; ok; ++j) {
                const int t = tile_of(j, leader, false);
                if (t < 0)
                    break;
                const int np = t % n_pairs, rest = t / n_pairs;
                const int mp = rest % m_pairs, l = rest / m_pairs;
                const int m0 = mp * 256 + 128 * (int)rank;
                const int nb = np * 256 + 128 * (int)rank;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (uint32_t)(it / S) & 1u;
                    if (!mbar_wait(empty0 + 8u * s, ph ^ 1u)) {
                        raise_fault(kFaultLoad);
                        ok = false;
                        break;
                    }
                    const uint32_t full = map_to_rank(bar0 + 8u * s, 0);
                    if (leader)
                        mbar_expect_tx(bar0 + 8u * s, kForm ? 2u * PairCfg::kBHalf : PairCfg::kPairTx);
                    const int kc = kb * BK;
                    if (kForm) {
                        // this CTA's z rows into its own A stage (z is [T, D]: one "layer")
                        mbar_expect_tx(aload0 + 8u * s, kABytes);
                        tma_load_3d(sA + s * kABytes, &tmA, kc, m0, 0, aload0 + 8u * s);
                    } else {
                        tma_load_3d_pair(sA + s * kABytes, &tmA, kc, m0, l, full);
                    }
                    if (kBmn) {
                        tma_load_3d_pair(sB + s * PairCfg::kBHalf, &tmB, nb, kc, l, full);
                        tma_load_3d_pair(sB + s * PairCfg::kBHalf + 8192u, &tmB, nb + 64, kc, l, full);
                    } else {
                        tma_load_3d_pair(sB + s * PairCfg::kBHalf, &tmB, kc, nb, l, full);
                    }
                    issued = it + 1;
                }
            }
        }
    } else if (kForm && warp == 1 && !leader) {
        // the peer's idle MMA thread forwards "A formed" to the leader, so
        // the forming warps never pay for a cluster-scope release
        if (lane == 0 && !skip) {
            const uint32_t peer_lead = map_to_rank(peer0, 0);
            int it = 0;
            bool ok = true;
            for (int j = 0; ok; ++j) {
                if (tile_of(j, false, false) < 0)
                    break;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    if (!mbar_wait(ready0 + 8u * s, (uint32_t)(it / S) & 1u)) {
                        raise_fault(kFaultMma);
                        ok = false;
                        break;
                    }
                    mbar_arrive_cluster(peer_lead + 8u * s);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int consumed = 0;
            if (!skip) {
                constexpr uint32_t idesc = make_idesc(256, 256, kBmn);
                int it = 0;
                bool ok = true;
                for (int j = 0; ok; ++j) {
                    const int t = tile_of(j, false, false);
                    if (t < 0)
                        break;
                    const int b = j & 1;
                    // both epilogues are done reading accumulator b (tile j - 2)
                    if (!mbar_wait_cluster(aempty0 + 8u * b, ((uint32_t)(j >> 1) & 1u) ^ 1u)) {
                        raise_fault(kFaultMma);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + 256u * (uint32_t)b;
                    for (int kb = 0; kb < nkb; ++kb, ++it) {
                        const int s = it % S;
                        const uint32_t ph = (uint32_t)(it / S) & 1u;
                        if (!mbar_wait(bar0 + 8u * s, ph) ||
                            (kForm && (!mbar_wait(ready0 + 8u * s, ph) ||
                                       !mbar_wait(peer0 + 8u * s, ph)))) {
                            raise_fault(kFaultMma);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a = sA + s * kABytes, bb = sB + s * PairCfg::kBHalf;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad = smem_desc_sw128(a + 32u * kk, 16u, 1024u);
                            const uint64_t bd = kBmn ? smem_desc_sw128(bb + 2048u * kk, 8192u, 1024u)
                                                     : smem_desc_sw128(bb + 32u * kk, 16u, 1024u);
                            mma_bf16_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                        }
                        mma_commit_pair(empty0 + 8u * s);
                        consumed = it + 1;
                    }
                    if (ok)
                        mma_commit_pair(afull0 + 8u * b);   // accumulator b holds tile j
                }
            }
            words[1] = (uint32_t)consumed;
            mma_commit_pair(done);
        }
        __syncwarp();
    } else if (kForm && warp >= 6) {
        // Forming warps: group grp (warps 6 + 4 grp ...) forms the stages it
        // with it % kPersistFormGroups == grp (the ring's stage count is a
        // multiple of the groups, so a stage always serves one group); thread
        // t of a group takes logical chunk c = t % 8 (8 columns) of rows
        // t / 8 + 16 j of this CTA's 128 rows.
        const int grp = (warp - 6) / kFormWarpsPerGroup;
        const int t8 = ((int)threadIdx.x - kThreads) % (32 * kFormWarpsPerGroup);
        const int c = t8 & 7, r0 = t8 >> 3;
        constexpr int kRowStep = 4 * kFormWarpsPerGroup;   // rows between one thread's rows
        int it = 0;
        bool ok = true;
        for (int j = 0; ok && !skip; ++j) {
            const int t = tile_of(j, false, true);
            if (t < 0)
                break;
            const int mp = t / n_pairs % m_pairs, l = t / n_pairs / m_pairs;
            const int m0 = mp * 256 + 128 * (int)rank;
            float rs[kFormRows];
#pragma unroll
            for (int jj = 0; jj < kFormRows; ++jj) {
                const int row = m0 + r0 + kRowStep * jj;
                rs[jj] = row < g.T ? __ldg(g.row_scale + row) : 0.0f;
            }
            const uint16_t *gain = g.col_gain ? g.col_gain + (int64_t)l * (nkb * BK) + 8 * c : nullptr;
            // the gains of this group's next stage of the tile are fetched
            // while the current one is formed, so no stage waits for them
            const int kb_first = ((grp - it) % kPersistFormGroups + kPersistFormGroups) % kPersistFormGroups;
            uint4 g_next = make_uint4(0, 0, 0, 0);
            if (gain && kb_first < nkb)
                g_next = __ldg(reinterpret_cast<const uint4 *>(gain + kb_first * BK));
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                if (it % kPersistFormGroups != grp)
                    continue;
                const int s = it % S;
                float gm[8];
                if (gain) {
                    unpack8f(g_next, gm);
                    if (kb + kPersistFormGroups < nkb)
                        g_next = __ldg(reinterpret_cast<const uint4 *>(gain + (kb + kPersistFormGroups) * BK));
                }
                if (!mbar_wait(aload0 + 8u * s, (uint32_t)(it / S) & 1u)) {
                    raise_fault(kFaultLoad);
                    ok = false;
                    break;
                }
                // all rows' chunks in flight, then formed, then written back;
                // rows r0 + kRowStep jj share r % 8 (kRowStep is a multiple of
                // 8), so their swizzled chunks sit kRowStep * 128 bytes apart
                static_assert(kRowStep % 8 == 0, "one swizzle phase for a thread's rows");
                const uint32_t base = sA + s * kABytes + r0 * 128 + ((c ^ (r0 & 7)) << 4);
                uint4 v[kFormRows];
#pragma unroll
                for (int jj = 0; jj < kFormRows; ++jj)
                    v[jj] = ld_shared_v4(base + 128u * kRowStep * jj);
#pragma unroll
                for (int jj = 0; jj < kFormRows; ++jj)
                    v[jj] = form_chunk(v[jj], rs[jj], gain ? gm : nullptr);
#pragma unroll
                for (int jj = 0; jj < kFormRows; ++jj)
                    st_shared_v4(base + 128u * kRowStep * jj, v[jj]);
                // generic-proxy writes, then visible to the tensor core
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_local(ready0 + 8u * s);
            }
        }
    } else {
        const int q = warp & 3;
        const uint32_t stage = sStage + (uint32_t)q * kStageRowsBytes;
        for (int j = 0; !skip; ++j) {
            const int t = tile_of(j, false, true);
            if (t < 0)
                break;
            const int b = j & 1;
            bool ok = mbar_wait(afull0 + 8u * b, (uint32_t)(j >> 1) & 1u);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                if (lane == 0)
                    raise_fault(kFaultAccum);
                break;
            }
            tc_fence_after();
            const int np = t % n_pairs, rest = t / n_pairs;
            const int mp = rest % m_pairs, l = rest / m_pairs;
            const int m0 = mp * 256 + 128 * (int)rank, n0 = np * 256;
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + 256u * (uint32_t)b;
            if (kFused)
                fused_store_tile<!kForm>(fs, g, tbase, l, m0 + 32 * q + lane, n0, stage, lane);
            else
                write_bf16_rows(g, tbase, stage, m0 + 32 * q, l, n0, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_release_cluster(map_to_rank(aempty0 + 8u * b, 0));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (!leader && warp == 0 && lane == 0)
        st_cluster_u32(map_to_rank(words_addr + 12u, 0), (uint32_t)issued);
    cluster_sync();
    if (warp == 0 && lane == 0 && leader) {
        // Both CTAs' loads land on the leader's barriers: after a fault, wait
        // for every stage either CTA issued before anyone frees smem.
        const int last = max(issued, (int)words[3]);
        for (int i = (int)words[1]; i < last; ++i)
            if (!mbar_wait_own(bar0 + 8u * (i % S), (uint32_t)(i / S) & 1u)) {
                raise_fault(kFaultDrain);
                break;
            }
    }
    if (kForm && warp == 0 && lane == 0)              // this CTA's own z loads
        for (int i = max(0, issued - S); i < issued; ++i)
            if (!mbar_wait_own(aload0 + 8u * (i % S), (uint32_t)(i / S) & 1u)) {
                raise_fault(kFaultDrain);
                break;
            }
    if (leader && warp == 1 && lane == 0 && !mbar_wait_own(done, 0u))
        raise_fault(kFaultDrain);
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host

template <int BN, bool kBmn>
cudaError_t launch_tile(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &g,
                        int n_tiles, int m_tiles, cudaStream_t stream) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(k2_project<BN, kBmn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Cfg<BN>::kSmem);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            configured[dev] = true;
    }
    const dim3 grid((unsigned)n_tiles, (unsigned)m_tiles, (unsigned)(g.L * g.splits));
    return launch_pdl(k2_project<BN, kBmn>, grid, dim3(kThreads), Cfg<BN>::kSmem, stream, 1, ma, mb, g);
}

template <bool kBmn, bool kFused, bool kTransform>
cudaError_t launch_pair(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &g,
                        const FusedStore &fs, int n_pairs, int m_pairs, cudaStream_t stream) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(k2_project_pair<kBmn, kFused, kTransform>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PairCfg::kSmem);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            configured[dev] = true;
    }
    const dim3 grid((unsigned)(2 * n_pairs), (unsigned)m_pairs, (unsigned)(g.L * g.splits));
    return launch_pdl(k2_project_pair<kBmn, kFused, kTransform>, grid,
                      dim3(pair_threads<kTransform>()), PairCfg::kSmem, stream, 2, ma, mb, g, fs);
}

// One CTA pair per two SMs (fewer when there are fewer tiles).
template <bool kBmn, bool kFused, bool kForm = false>
cudaError_t launch_pair_persistent(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &g,
                                   const FusedStore &fs, int n_pairs, int m_pairs, int tile_limit,
                                   unsigned int *tile_ctr, cudaStream_t stream) {
    static int sms[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    int n_sms = dev < 64 ? sms[dev] : 0;
    if (n_sms == 0) {
        e = cudaFuncSetAttribute(k2_project_pair_persistent<kBmn, kFused, kForm>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PersistCfg::kSmem);
        if (e != cudaSuccess)
            return e;
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            sms[dev] = n_sms;
    }
    const int64_t tiles = std::min<int64_t>((int64_t)g.L * m_pairs * n_pairs, tile_limit);
    const int pairs = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, n_sms / 2));
    return launch_pdl(k2_project_pair_persistent<kBmn, kFused, kForm>, dim3((unsigned)(2 * pairs)),
                      dim3(persist_threads(kForm)), PersistCfg::kSmem, stream, 2, ma, mb, g, fs,
                      n_pairs, m_pairs, tile_limit, tile_ctr);
}

}  // namespace

ProjectPlan plan_kv_project(int32_t L, int64_t T, int32_t D, int32_t N, int num_sms,
                            size_t workspace_bytes, bool allow_tail)
{
    ProjectPlan p{};
    p.tile_ctr_offset = -1;
    if (T <= 0 || L <= 0 || D < BK || N < 128 || num_sms < 1) {
        // nothing to launch: single CTAs without splits, no workspace
        p.bn = 128;
        p.splits = p.tail_splits = 1;
        p.kb_per_split = p.tail_kb_per_split = std::max(1, D / BK);
        return p;
    }
    // 256-wide N tiles where there are rows to fill them; with one 128-row
    // block (T <= 128) the projection streams W at too few bytes of work per
    // byte to be tensor-bound, so 128-wide tiles put twice the CTAs (SMs) on
    // reading W (workload 1: 25.1 -> 23.1-23.4 us a step)
    p.bn = (N % 256 == 0 && T > BM) ? 256 : 128;
    // CTA pairs need two 128-row halves with work and 256-wide N tiles.
    p.pair = p.bn == 256 && T > BM;
    const int kb_total = D / BK;
    const int64_t tiles = p.pair ? 2 * (int64_t)L * ((T + 255) / 256) * (N / 256)
                                 : (int64_t)L * ((T + BM - 1) / BM) * (N / p.bn);
    int splits = 1;
    if (tiles < num_sms) {
        splits = (int)(num_sms / tiles);
        // >= 8 K blocks per split: more, shorter splits only add partials
        // for the reduction to read (32 splits of 4 blocks measured 15 %
        // slower than 16 of 8 at T = 64)
        splits = std::min(splits, std::max(1, kb_total / 8));
    }
    const size_t per_split = (size_t)L * (size_t)T * (size_t)N * sizeof(float);
    while (splits > 1 && (size_t)splits * per_split > workspace_bytes)
        --splits;
    p.kb_per_split = (kb_total + splits - 1) / splits;
    p.splits = (kb_total + p.kb_per_split - 1) / p.kb_per_split;   // no empty split
    p.workspace = p.splits > 1 ? (size_t)p.splits * per_split : 0;
    p.tail_splits = 1;
    p.tail_kb_per_split = kb_total;
    p.tile_ctr_offset = -1;
    if (p.pair && p.splits == 1) {
        // Persistent pairs take tiles round-robin, so a last wave of rem <
        // P tiles costs a whole tile time.  Its tiles (rounded up to whole
        // 256-row blocks, all in the last layer) can instead run split over
        // the idle pairs: (full waves) + 1 / s tile times plus a fixed cost
        // (fill, partials, reduce-and-store: about 20 K blocks' time).
        const int64_t n_pairs = N / 256, m_pairs = (T + 255) / 256;
        const int64_t P = std::max(1, num_sms / 2);
        const int64_t rem = tiles / 2 % P;               // `tiles` counts CTAs here
        const int64_t tail = (rem + n_pairs - 1) / n_pairs * n_pairs;
        if (allow_tail && tiles / 2 > P && rem > 0 && tail <= m_pairs * n_pairs && tail < P) {
            int s = (int)std::min<int64_t>(P / tail, kb_total / 8);
            const int64_t row0 = (m_pairs - tail / n_pairs) * 256;
            const size_t per_tail_split = (size_t)(T - row0) * (size_t)N * sizeof(float);
            while (s > 1 && (size_t)s * per_tail_split > workspace_bytes)
                --s;
            const int64_t waves = (tiles / 2 + P - 1) / P;
            const int64_t full_waves = (tiles / 2 - tail + P - 1) / P;
            if (s >= 2 && (double)full_waves + 1.0 / s + 20.0 / kb_total < (double)waves) {
                p.tail_tiles = tail;
                p.tail_row0 = row0;
                p.tail_kb_per_split = (kb_total + s - 1) / s;
                p.tail_splits = (kb_total + p.tail_kb_per_split - 1) / p.tail_kb_per_split;
                p.workspace = (size_t)p.tail_splits * per_tail_split;
            }
        }
        // Eight rounds of tiles or more: pairs take tiles from a counter in
        // the workspace (after the tail's partials), when it has room.  With
        // fewer rounds the pairs do not drift apart far enough to lose their
        // shared A reads in L2 (workload 3, 3 rounds: 11 % more DRAM bytes
        // than the operands; workload 5, 54 rounds: 2.5 times), and the fixed
        // order keeps the launch overlapping the previous kernel's end.
        const int64_t persistent_tiles = tiles / 2 - p.tail_tiles;
        const size_t off = (p.workspace + 255) / 256 * 256;
        if (persistent_tiles >= 8 * P && persistent_tiles < kMaxDynTiles &&
            off + 256 <= workspace_bytes) {
            p.tile_ctr_offset = (int64_t)off;
            p.workspace = off + 256;
        }
    }
    return p;
}

namespace {

// Tensor maps and kernel arguments of one projection.
bool project_setup(const uint16_t *normed, const uint16_t *W, bool w_nk, uint16_t *out, int32_t L,
                   int64_t T, int32_t D, int32_t N, const ProjectPlan &plan, float *ws,
                   CUtensorMap *ma, CUtensorMap *mb, GemmArgs *g, const char **why) {
    if (!make_map(ma, normed, (uint64_t)D, (uint64_t)T, (uint64_t)L, BK, BM)) {
        *why = "tensor map of the normed rows could not be encoded";
        return false;
    }
    const uint32_t b_rows = plan.pair ? 128u : (uint32_t)plan.bn;   // K-major B rows per CTA
    const bool ok_b = w_nk ? make_map(mb, W, (uint64_t)D, (uint64_t)N, (uint64_t)L, BK, b_rows)
                           : make_map(mb, W, (uint64_t)N, (uint64_t)D, (uint64_t)L, 64, BK);
    if (!ok_b) {
        *why = "tensor map of the weights could not be encoded";
        return false;
    }
    g->T = (int32_t)T;
    g->N = N;
    g->L = L;
    g->kb_total = D / BK;
    g->kb_per_split = plan.kb_per_split;
    g->splits = plan.splits;
    g->out = out;
    g->partial = ws;
    g->row_scale = nullptr;
    g->col_gain = nullptr;
    return true;
}

// The GEMM kernel of a plan (no split-K reduction).
template <bool kFused>
cudaError_t launch_gemm(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &g,
                        const FusedStore &fs, bool w_nk, const ProjectPlan &plan, int64_t T,
                        int32_t N, cudaStream_t stream) {
    if (plan.pair && plan.splits == 1) {       // persistent pairs, epilogue under the next mainloop
        const int n_pairs = N / 256, m_pairs = (int)((T + 255) / 256);
        const int limit = (int)((int64_t)g.L * m_pairs * n_pairs - plan.tail_tiles);
        unsigned int *ctr = nullptr;
        if (plan.tile_ctr_offset >= 0 && g.partial != nullptr) {
            ctr = reinterpret_cast<unsigned int *>(reinterpret_cast<char *>(g.partial) +
                                                   plan.tile_ctr_offset);
            if (!plan.ctr_zeroed) {
                const cudaError_t e = cudaMemsetAsync(ctr, 0, sizeof(unsigned int), stream);
                if (e != cudaSuccess)
                    return e;
            }
        }
        return w_nk ? launch_pair_persistent<false, kFused>(ma, mb, g, fs, n_pairs, m_pairs, limit, ctr, stream)
                    : launch_pair_persistent<true, kFused>(ma, mb, g, fs, n_pairs, m_pairs, limit, ctr, stream);
    }
    if (plan.pair)
        return w_nk ? launch_pair<false, kFused, false>(ma, mb, g, fs, N / 256, (int)((T + 255) / 256), stream)
                    : launch_pair<true, kFused, false>(ma, mb, g, fs, N / 256, (int)((T + 255) / 256), stream);
    const int n_tiles = N / plan.bn;
    const int m_tiles = (int)((T + BM - 1) / BM);
    if (plan.bn == 256)
        return w_nk ? launch_tile<256, false>(ma, mb, g, n_tiles, m_tiles, stream)
                    : launch_tile<256, true>(ma, mb, g, n_tiles, m_tiles, stream);
    return w_nk ? launch_tile<128, false>(ma, mb, g, n_tiles, m_tiles, stream)
                : launch_tile<128, true>(ma, mb, g, n_tiles, m_tiles, stream);
}

cudaError_t launch_reduce(const float *ws, uint16_t *out, int64_t count, int splits,
                          cudaStream_t stream) {
    const int64_t blocks = std::min<int64_t>((count / 8 + 255) / 256, 152 * 16);
    return launch_pdl(k2_splitk_reduce, dim3((unsigned)blocks), dim3(256), 0, stream, 1, ws, out,
                      count, splits);
}

// The tail of a persistent plan: rows tail_row0 .. T-1 of the last layer as
// a one-layer split-K problem of CTA pairs writing FP32 partials to ws
// ([tail_splits, T - tail_row0, N]); the caller then reduces them.
cudaError_t launch_tail_partials(const uint16_t *normed, const uint16_t *W, bool w_nk, int32_t L,
                                 int64_t T, int32_t D, int32_t N, const ProjectPlan &plan,
                                 float *ws, cudaStream_t stream, const char **why) {
    const int64_t rows = T - plan.tail_row0;
    const uint16_t *a = normed + ((int64_t)(L - 1) * T + plan.tail_row0) * D;
    const uint16_t *b = W + (int64_t)(L - 1) * D * N;
    CUtensorMap ma, mb;
    if (!make_map(&ma, a, (uint64_t)D, (uint64_t)rows, 1, BK, BM)) {
        *why = "tensor map of the tail rows could not be encoded";
        return cudaErrorInvalidValue;
    }
    const bool ok_b = w_nk ? make_map(&mb, b, (uint64_t)D, (uint64_t)N, 1, BK, 128)
                           : make_map(&mb, b, (uint64_t)N, (uint64_t)D, 1, 64, BK);
    if (!ok_b) {
        *why = "tensor map of the last layer's weights could not be encoded";
        return cudaErrorInvalidValue;
    }
    GemmArgs g{};
    g.T = (int32_t)rows;
    g.N = N;
    g.L = 1;
    g.kb_total = D / BK;
    g.kb_per_split = plan.tail_kb_per_split;
    g.splits = plan.tail_splits;
    g.out = nullptr;
    g.partial = ws;
    g.row_scale = nullptr;
    g.col_gain = nullptr;
    FusedStore none{};
    *why = "tail projection launch";
    const int m_pairs = (int)((rows + 255) / 256);
    return w_nk ? launch_pair<false, false, false>(ma, mb, g, none, N / 256, m_pairs, stream)
                : launch_pair<true, false, false>(ma, mb, g, none, N / 256, m_pairs, stream);
}

}  // namespace

cudaError_t launch_kv_project(const uint16_t *normed, const uint16_t *W, bool w_nk, uint16_t *out,
                              int32_t L, int64_t T, int32_t D, int32_t N, const ProjectPlan &plan,
                              float *ws, cudaStream_t stream, const char **why)
{
    CUtensorMap ma, mb;
    GemmArgs g;
    if (!project_setup(normed, W, w_nk, out, L, T, D, N, plan, ws, &ma, &mb, &g, why))
        return cudaErrorInvalidValue;
    FusedStore none{};
    cudaError_t e = launch_gemm<false>(ma, mb, g, none, w_nk, plan, T, N, stream);
    if (e != cudaSuccess)
        return e;
    if (plan.tail_tiles > 0) {
        // the last layer's tail rows: split partials, then their reduction
        e = launch_tail_partials(normed, W, w_nk, L, T, D, N, plan, ws, stream, why);
        if (e != cudaSuccess)
            return e;
        const int64_t rows = T - plan.tail_row0;
        return launch_reduce(ws, out + ((int64_t)(L - 1) * T + plan.tail_row0) * N, rows * N,
                             plan.tail_splits, stream);
    }
    if (plan.splits == 1)
        return e;
    return launch_reduce(ws, out, (int64_t)L * T * N, plan.splits, stream);
}

cudaError_t launch_kv_project_store(const uint16_t *normed, const uint16_t *W, bool w_nk,
                                    int32_t L, int64_t T, int32_t D, int32_t N,
                                    const ProjectPlan &plan, float *ws, const FusedStore &fs,
                                    cudaStream_t stream, const char **why)
{
    CUtensorMap ma, mb;
    GemmArgs g;
    if (!project_setup(normed, W, w_nk, fs.kv_out, L, T, D, N, plan, ws, &ma, &mb, &g, why))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (plan.splits > 1) {
        // partials, then one pass that reduces and stores
        e = launch_gemm<false>(ma, mb, g, fs, w_nk, plan, T, N, stream);
        if (e != cudaSuccess)
            return e;
        *why = "reduce-and-store launch";
        return launch_reduce_store(fs, ws, plan.splits, L, (int32_t)T, stream);
    }
    if (plan.pair) {                               // the epilogue stores
        e = launch_gemm<true>(ma, mb, g, fs, w_nk, plan, T, N, stream);
        if (e != cudaSuccess || plan.tail_tiles == 0)
            return e;
        // the last layer's tail rows: split partials, then reduce-and-store
        // them as a one-layer problem
        e = launch_tail_partials(normed, W, w_nk, L, T, D, N, plan, ws, stream, why);
        if (e != cudaSuccess)
            return e;
        const int64_t row0 = plan.tail_row0, rows = T - row0;
        const int32_t last = L - 1;
        FusedStore ts = fs;
        const int64_t kept = std::min<int64_t>(std::max<int64_t>(fs.rows[last] - row0, 0), rows);
        ts.slots[0] = kept > 0 ? fs.slots[last] + row0 : nullptr;
        ts.caches[0] = fs.caches[last];
        ts.rows[0] = (int32_t)kept;
        for (int i = 1; i < kMaxFusedLayers; ++i) {
            ts.slots[i] = nullptr;
            ts.caches[i] = nullptr;
            ts.rows[i] = 0;
        }
        if (fs.positions != nullptr)
            ts.positions = fs.positions + row0;
        if (fs.kv_out != nullptr)
            ts.kv_out = fs.kv_out + ((int64_t)last * T + row0) * N;
        *why = "tail reduce-and-store launch";
        return launch_reduce_store(ts, ws, plan.tail_splits, 1, (int32_t)rows, stream);
    }
    // single CTAs without a split: the projection lands in kv_out, then the
    // store kernel reads it (8 layers per launch)
    if (fs.kv_out == nullptr) {
        *why = "this size needs kv_out (the projection is stored from it)";
        return cudaErrorInvalidValue;
    }
    e = launch_gemm<false>(ma, mb, g, fs, w_nk, plan, T, N, stream);
    if (e != cudaSuccess)
        return e;
    for (int32_t first = 0; first < L; first += kMaxLayersPerLaunch) {
        const int32_t n = std::min(kMaxLayersPerLaunch, L - first);
        StoreLaunch p{};
        bool any = false;
        for (int32_t i = 0; i < n; ++i) {
            p.slots[i] = fs.rows[first + i] > 0 ? fs.slots[first + i] : nullptr;
            p.caches[i] = fs.caches[first + i];
            p.rows[i] = fs.rows[first + i];
            any = any || p.slots[i] != nullptr;
            if (p.slots[i])
                p.grid_rows = std::max(p.grid_rows, p.rows[i]);
        }
        if (!any)
            continue;
        p.k = fs.kv_out + (int64_t)first * T * N;
        p.v = p.k + 64 * fs.H;
        p.k_layer_stride = p.v_layer_stride = T * N;
        p.k_row_stride = p.v_row_stride = N;
        p.positions = fs.positions;
        p.cos_sin = fs.cos_sin;
        p.max_position = fs.max_position;
        p.capacity = fs.capacity;
        p.block_size = fs.block_size;
        p.eps = fs.eps;
        p.err = fs.err;
        e = launch_kv_store(p, fs.H, n, stream);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t launch_kv_from_rows(const uint16_t *z, const float *r2, int64_t T,
                                const uint16_t *pre_w, const uint16_t *W, bool w_nk, int32_t L,
                                int32_t N, const ProjectPlan &plan, float *ws, const FusedStore &fs,
                                cudaStream_t stream, const char **why)
{
    constexpr int D = kHidden;
    CUtensorMap ma, mb;
    GemmArgs g;
    if (!project_setup(z, W, w_nk, fs.kv_out, L, T, D, N, plan, ws, &ma, &mb, &g, why))
        return cudaErrorInvalidValue;
    // A is z [T, D] (one "layer"), formed per layer in shared memory
    if (!make_map(&ma, z, (uint64_t)D, (uint64_t)T, 1, BK, BM)) {
        *why = "tensor map of the hidden-norm rows could not be encoded";
        return cudaErrorInvalidValue;
    }
    g.row_scale = r2;
    g.col_gain = pre_w;
    const int n_pairs = N / 256, m_pairs = (int)((T + 255) / 256);
    *why = "fused projection launch";
    if (plan.splits == 1 && plan.tile_ctr_offset >= 0 && ws != nullptr) {
        // eight rounds of tiles or more: persistent pairs forming A in shared
        // memory (2 groups of 4 forming warps), every tile in this launch, the
        // tiles taken from the workspace's counter
        unsigned int *ctr =
            reinterpret_cast<unsigned int *>(reinterpret_cast<char *>(ws) + plan.tile_ctr_offset);
        const cudaError_t e = cudaMemsetAsync(ctr, 0, sizeof(unsigned int), stream);
        if (e != cudaSuccess)
            return e;
        const int limit = L * m_pairs * n_pairs;
        return w_nk ? launch_pair_persistent<false, true, true>(ma, mb, g, fs, n_pairs, m_pairs, limit,
                                                                ctr, stream)
                    : launch_pair_persistent<true, true, true>(ma, mb, g, fs, n_pairs, m_pairs, limit,
                                                               ctr, stream);
    }
    if (plan.splits == 1)      // one CTA pair per tile, 3 groups of 4 forming warps
        return w_nk ? launch_pair<false, true, true>(ma, mb, g, fs, n_pairs, m_pairs, stream)
                    : launch_pair<true, true, true>(ma, mb, g, fs, n_pairs, m_pairs, stream);
    cudaError_t e = w_nk ? launch_pair<false, false, true>(ma, mb, g, fs, n_pairs, m_pairs, stream)
                         : launch_pair<true, false, true>(ma, mb, g, fs, n_pairs, m_pairs, stream);
    if (e != cudaSuccess)
        return e;
    *why = "reduce-and-store launch";
    return launch_reduce_store(fs, ws, plan.splits, L, (int32_t)T, stream);
}

cudaError_t read_project_faults(uint32_t *flags, bool clear)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return e;
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_project_faults, sizeof v);
    if (e != cudaSuccess)
        return e;
    *flags = v;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_project_faults, &zero, sizeof zero);
    }
    return e;
}

}  // namespace rc
