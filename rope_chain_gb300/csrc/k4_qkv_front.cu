// K4: the decode QKV front -- one draft layer's QKV projection of 1 to 16
// tokens, the QK-norm and GPT-J RoPE of its Q and K heads, and the insert of
// K and V into the layer's paged cache, in one kernel.
//
// Page "vllm.models.muse_spark.nvidia.specialized_decode.runtime.draft":
// _fused_qkv_projection (one call per layer: hidden states, the qkv_proj
// weight [Nqkv, D], positions, the cos|sin table, the slot mapping, the KV
// cache and rms_norm_eps), _attention (the output row splits as
// [Q | K | V | O-gate], q_size = 64 * num_heads, kv_size = 64 *
// num_kv_heads) and may_fuse_qkv_front (1 to 16 tokens, 64-wide heads).  The
// per-head norm and rotation are the context store's (weightless RMSNorm in
// the lane-pair butterfly order, bf16, then GPT-J RoPE).
//
// GB300 design.  With at most 16 tokens the projection streams the weight
// once and does almost no arithmetic per byte, so the kernel is built around
// reading W at HBM speed:
//   * operands swapped: each CTA owns 128 output columns (128 rows of W, the
//     MMA's M) and all tokens (the MMA's N = 16; TMA fills token rows past M
//     with zeros): tcgen05.mma 128 x 16 x 16, the accumulator is 16 TMEM
//     columns;
//   * warp 0 streams 18 KiB stages (16 KiB of W, 2 KiB of hidden states)
//     through a 10-deep TMA ring, warp 1 issues the MMAs;
//   * when there are few column tiles, a cluster of 2 CTAs splits K in
//     halves; the upper half's FP32 accumulator crosses to the lower CTA's
//     shared memory (DSMEM) and is added after it (lower K first, a fixed
//     order);
//   * the epilogue rounds the projection to bf16 into a token-major staging
//     tile, then one warp per (token, head) applies the context store's
//     lane-pair K-norm and RoPE to Q and K heads, writes the output row and
//     inserts K and V.
// Every wait is bounded; on timeout the kernel raises a sticky fault bit,
// skips its remaining work and drains its own copies.
#include "rc_internal.cuh"
#include "rc_tcgen05.cuh"

#include <algorithm>

namespace rc {

__device__ unsigned int g_front_faults;

namespace {

constexpr int kBM = 128;                        // W rows (output columns) per CTA
constexpr int kBK = 64;                         // one 128-byte swizzle row of bf16
constexpr int kTok = 16;                        // tokens per MMA (N)
constexpr int kStages = 10;
constexpr int kThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;     // 16 KiB
constexpr uint32_t kBBytes = kTok * kBK * 2;    // 2 KiB
constexpr uint32_t kRedStride = 80;             // bytes per column of the DSMEM partial
constexpr uint32_t kRedBytes = kBM * kRedStride;
constexpr uint32_t kStgBytes = kTok * kBM * 2;  // bf16 [16 tokens][128 columns]
// per token: position, slot, and its cos|sin table row (64 bf16)
constexpr uint32_t kTokBytes = kTok * 8 * 2 + kTok * kHeadDim * 2;
constexpr size_t kSmem = 1024 + (size_t)kStages * (kABytes + kBBytes) + kRedBytes + kStgBytes +
                         kTokBytes + 256;

// Per-token operands of the epilogue, fetched while the weight streams.
struct TokenInfo {
    int64_t pos[kTok];
    int64_t slot[kTok];
    uint16_t cs[kTok][kHeadDim];       // the token's table row: cos 0..31, sin 32..63
};
static_assert(sizeof(TokenInfo) == kTokBytes, "token block size");

enum : unsigned { kFaultLoad = 1u, kFaultMma = 2u, kFaultAccum = 4u, kFaultDrain = 8u };

__device__ __forceinline__ void raise_fault(unsigned bit) { atomicOr(&g_front_faults, bit); }
__device__ __forceinline__ bool faulted() {
    return *reinterpret_cast<volatile unsigned int *>(&g_front_faults) != 0u;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_wait_flag(bar, parity, &g_front_faults);
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
    return d;
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct FrontArgs {
    int32_t M;                   // tokens, 1..16
    int32_t N;                   // 64 * (2 * num_heads + 2 * num_kv_heads)
    int32_t num_heads, num_kv_heads;
    int32_t kb_total, kb_per_split;
    const int64_t *positions;    // [M] (read with a table)
    const uint16_t *cos_sin;     // bf16 [max_position, 64] or NULL
    int64_t max_position;
    const int64_t *slots;        // [M] or NULL
    uint16_t *cache;             // bf16 [num_blocks, num_kv_heads, block_size, 128]
    int64_t capacity;            // num_blocks * block_size
    int32_t block_size;
    float eps;
    uint16_t *out;               // bf16 [M, N]
    uint16_t *raw;               // bf16 [M, N] projection, or NULL
    int32_t *err;
};

// One (token, head) of the epilogue, a whole warp: lane j holds the pair
// (2j, 2j+1) of head column block `col` of token m; tk holds the token's
// position, slot and table row.
__device__ __forceinline__ void front_head(const FrontArgs &a, const TokenInfo &tk, int m, int col,
                                           uint32_t word, int lane) {
    const int gh = col >> 6;                        // head index in [Q | K | V | gate]
    const int nq = a.num_heads, nkv = a.num_kv_heads;
    const int64_t at = (int64_t)m * a.N + col;
    if (a.raw != nullptr)
        reinterpret_cast<uint32_t *>(a.raw + at)[lane] = word;
    int64_t pos = 0;
    bool bad_pos = false;
    if (a.cos_sin != nullptr) {
        pos = tk.pos[m];
        bad_pos = pos < 0 || pos >= a.max_position;
    }
    const int64_t slot = a.slots != nullptr ? tk.slot[m] : -1;
    const bool insert = slot >= 0 && slot < a.capacity && !bad_pos;
    uint32_t *dst = nullptr;
    if (insert && gh >= nq && gh < nq + 2 * nkv) {
        // Slots of a cache fit 32 bits (checked on the host).
        const uint32_t bs = (uint32_t)a.block_size;
        const uint32_t blk = (uint32_t)slot / bs;
        const uint32_t page = (uint32_t)slot - blk * bs;
        const int h = gh < nq + nkv ? gh - nq : gh - nq - nkv;
        dst = reinterpret_cast<uint32_t *>(a.cache) +
              (((int64_t)blk * nkv + h) * bs + page) * kHeadDim + (gh < nq + nkv ? 0 : kHeadDim / 2);
    }
    uint32_t o = word;
    if (gh < nq + nkv) {                            // Q or K: QK-norm, then RoPE
        if (a.cos_sin != nullptr && !bad_pos) {
            const float c = __uint_as_float((uint32_t)tk.cs[m][lane] << 16);
            const float s = __uint_as_float((uint32_t)tk.cs[m][kHeadDim / 2 + lane] << 16);
            o = knorm_rope_lane<true>(bf16_lo(word), bf16_hi(word), c, s, a.eps);
        } else {
            o = knorm_rope_lane<false>(bf16_lo(word), bf16_hi(word), 1.0f, 0.0f, a.eps);
        }
    }
    reinterpret_cast<uint32_t *>(a.out + at)[lane] = o;
    if (dst != nullptr)
        dst[lane] = o;                              // K' (or V, which passes through)
}

__global__ void __launch_bounds__(kThreads, 1)
k4_qkv_front(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
             const __grid_constant__ FrontArgs a, int ksplit)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + kStages * kABytes;
    const uint32_t sRed = sB + kStages * kBBytes;   // the upper K half's FP32 partial
    const uint32_t sStg = sRed + kRedBytes;         // bf16 [16 tokens][128 columns]
    const uint32_t sTok = sStg + kStgBytes;         // TokenInfo
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * (kABytes + kBBytes) + kRedBytes +
                                                  kStgBytes + kTokBytes);
    TokenInfo &tk = *reinterpret_cast<TokenInfo *>(smem + (sTok - sA));
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8u * kStages;
    const uint32_t accum = full0 + 16u * kStages;
    // words[0]: TMEM base; [1]: the partner's partial is valid (set by rank 1
    // in rank 0); [2]: skip (a fault was raised before this launch); [3..6]:
    // epilogue warp q's accumulator arrived
    volatile uint32_t *words = reinterpret_cast<volatile uint32_t *>(bars + 2 * kStages + 1);
    const uint32_t words_addr = smem_u32((const void *)words);

    const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ksplit > 1 ? cluster_rank() : 0u;
    const int n0 = (int)(blockIdx.x / (unsigned)ksplit) * kBM;
    const int kb0 = (int)rank * a.kb_per_split;
    const int nkb = max(0, min(a.kb_per_split, a.kb_total - kb0));
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        mbar_init(accum, 1);
        words[1] = 0u;
        // one skip decision for the CTA, read before pdl_wait: a fault raised
        // by a kernel still finishing just before this one can be missed
        words[2] = faulted() ? 1u : 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmH);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(words_addr), "r"(32) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    if (ksplit > 1)
        cluster_barrier();                          // barriers initialised pair-wide
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = words[0];
    const bool skip = words[2] != 0u;
    pdl_wait();                                     // hidden states and caches of earlier kernels

    int issued = 0;
    if (warp == 0) {
        if (lane == 0 && !skip) {
            for (int i = 0; i < nkb; ++i) {
                const int s = i % kStages;
                if (!mbar_wait(empty0 + 8u * s, ((uint32_t)(i / kStages) & 1u) ^ 1u)) {
                    raise_fault(kFaultLoad);
                    break;
                }
                mbar_expect_tx(full0 + 8u * s, kABytes + kBBytes);
                const int kc = (kb0 + i) * kBK;
                tma_load_3d(sA + s * kABytes, &tmW, kc, n0, 0, full0 + 8u * s);
                tma_load_3d(sB + s * kBBytes, &tmH, kc, 0, 0, full0 + 8u * s);
                issued = i + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (!skip) {
                constexpr uint32_t idesc = make_idesc(kBM, kTok, false);
                for (int i = 0; i < nkb; ++i) {
                    const int s = i % kStages;
                    if (!mbar_wait(full0 + 8u * s, (uint32_t)(i / kStages) & 1u)) {
                        raise_fault(kFaultMma);
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(sA + s * kABytes + 32u * kk, 16u, 1024u);
                        const uint64_t bd = smem_desc_sw128(sB + s * kBBytes + 32u * kk, 16u, 1024u);
                        mma_bf16(tmem, ad, bd, idesc, (i | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty0 + 8u * s);
                }
            }
            mma_commit(accum);
        }
        __syncwarp();
    }

    // Epilogue part 1: the accumulator to registers (warp q owns TMEM lanes
    // = W rows 32q ... 32q + 31).  An empty K range (D smaller than the
    // split) leaves the accumulator unwritten: it counts as zeros.
    const int q = warp & 3;
    uint32_t acc[16];
    if (warp >= 2) {
        // While the weight streams: each token's position, slot and table
        // row into shared memory for the epilogue (the CTA that stores)
        if (rank == 0 && !skip) {
            for (int m = warp - 2; m < a.M; m += 4) {
                const int64_t pos = a.cos_sin != nullptr ? __ldg(a.positions + m) : 0;
                if (lane == 0) {
                    tk.pos[m] = pos;
                    tk.slot[m] = a.slots != nullptr ? __ldg(a.slots + m) : -1;
                }
                if (a.cos_sin != nullptr) {
                    const bool bad = pos < 0 || pos >= a.max_position;
                    const unsigned short *row =
                        reinterpret_cast<const unsigned short *>(a.cos_sin) + (bad ? 0 : pos) * kHeadDim;
                    tk.cs[m][lane] = __ldg(row + lane);
                    tk.cs[m][kHeadDim / 2 + lane] = __ldg(row + kHeadDim / 2 + lane);
                }
            }
        }
        bool ok = !skip && mbar_wait(accum, 0u);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok && !skip && lane == 0)
            raise_fault(kFaultAccum);
        if (lane == 0)
            words[3 + q] = ok ? 1u : 0u;
        if (ok && nkb > 0) {
            tc_fence_after();
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16), acc);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                acc[j] = 0u;
        }
        if (ksplit > 1 && rank == 1 && ok) {
            // the upper K half's partial into the lower CTA's shared memory
            const uint32_t dst = map_rank(sRed + (uint32_t)(32 * q + lane) * kRedStride, 0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st_cluster_v4(dst + 16u * j, acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
            if (warp == 2 && lane == 0)
                st_cluster_u32(map_rank(words_addr + 4u, 0), 1u);
        }
    }
    if (ksplit > 1)
        cluster_barrier();                          // the partial is visible to rank 0
    else
        __syncthreads();
    // CTA-uniform: every epilogue warp saw the accumulator, and the partner's
    // partial arrived
    const bool store = rank == 0 && words[3] != 0u && words[4] != 0u && words[5] != 0u &&
                       words[6] != 0u && (ksplit == 1 || words[1] != 0u);

    // Epilogue part 2 (rank 0): the sum in K order, rounded to bf16, staged
    // token-major, then one warp per (token, head).
    uint16_t *stg = reinterpret_cast<uint16_t *>(smem + (sStg - sA));
    if (store && warp >= 2) {
        const int col = 32 * q + lane;              // this thread's W row in the tile
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            v[j] = __uint_as_float(acc[j]);
        if (ksplit > 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 p = ld_shared_v4(sRed + (uint32_t)col * kRedStride + 16u * j);
                v[4 * j] = __fadd_rn(v[4 * j], __uint_as_float(p.x));
                v[4 * j + 1] = __fadd_rn(v[4 * j + 1], __uint_as_float(p.y));
                v[4 * j + 2] = __fadd_rn(v[4 * j + 2], __uint_as_float(p.z));
                v[4 * j + 3] = __fadd_rn(v[4 * j + 3], __uint_as_float(p.w));
            }
        }
#pragma unroll
        for (int m = 0; m < kTok; ++m)
            stg[m * kBM + col] = __bfloat16_as_ushort(__float2bfloat16_rn(v[m]));
    }
    if (store)
        __syncthreads();                            // the staging tile is complete
    if (store) {
        // all six warps take (token, head) items
        for (int item = warp; item < kTok * (kBM / kHeadDim); item += kThreads / 32) {
            const int m = item >> 1, hh = item & 1;
            if (m >= a.M)
                break;
            const uint32_t word = reinterpret_cast<const uint32_t *>(stg + m * kBM + hh * kHeadDim)[lane];
            front_head(a, tk, m, n0 + hh * kHeadDim, word, lane);
            if (n0 == 0 && hh == 0 && lane == 0 && a.err != nullptr) {
                // one count per token: the tile of column 0
                const int64_t slot = a.slots != nullptr ? tk.slot[m] : -1;
                bool bad = slot >= a.capacity;
                if (a.cos_sin != nullptr) {
                    const int64_t pos = tk.pos[m];
                    bad = bad || pos < 0 || pos >= a.max_position;
                }
                if (bad)
                    atomicAdd(a.err, 1);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        // every load this CTA issued has landed before smem is freed (the
        // last phase of each stage; all earlier ones were consumed)
        for (int i = max(0, issued - kStages); i < issued; ++i)
            if (!mbar_wait_own(full0 + 8u * (i % kStages), (uint32_t)(i / kStages) & 1u)) {
                raise_fault(kFaultDrain);
                break;
            }
    }
    if (warp == 1 && lane == 0 && !mbar_wait_own(accum, 0u))
        raise_fault(kFaultDrain);
    __syncwarp();
    tc_fence_before();
    if (ksplit > 1)
        cluster_barrier();
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32)
                     : "memory");
    }
}

}  // namespace

cudaError_t launch_qkv_front(const uint16_t *hidden, int32_t M, int32_t D, const uint16_t *W,
                             int32_t num_heads, int32_t num_kv_heads, const int64_t *positions,
                             const uint16_t *cos_sin, int64_t max_position, const int64_t *slots,
                             uint16_t *cache, int32_t num_blocks, int32_t block_size, float eps,
                             uint16_t *out, uint16_t *raw, int32_t *err, int num_sms,
                             cudaStream_t stream, const char **why)
{
    const int32_t N = kHeadDim * (2 * num_heads + 2 * num_kv_heads);
    CUtensorMap mw, mh;
    if (!make_map(&mw, W, (uint64_t)D, (uint64_t)N, 1, kBK, kBM) ||
        !make_map(&mh, hidden, (uint64_t)D, (uint64_t)M, 1, kBK, kTok)) {
        *why = "tensor maps of the weight or the hidden states could not be encoded";
        return cudaErrorInvalidValue;
    }
    FrontArgs a{};
    a.M = M;
    a.N = N;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.kb_total = D / kBK;
    const int n_tiles = N / kBM;
    const int ksplit = (2 * n_tiles <= num_sms && a.kb_total >= 2) ? 2 : 1;
    a.kb_per_split = (a.kb_total + ksplit - 1) / ksplit;
    a.positions = positions;
    a.cos_sin = cos_sin;
    a.max_position = max_position;
    a.slots = slots;
    a.cache = cache;
    a.capacity = (int64_t)num_blocks * block_size;
    a.block_size = block_size;
    a.eps = eps;
    a.out = out;
    a.raw = raw;
    a.err = err;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(k4_qkv_front, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            configured[dev] = true;
    }
    *why = "QKV front launch";
    return launch_pdl(k4_qkv_front, dim3((unsigned)(n_tiles * ksplit)), dim3(kThreads), kSmem, stream,
                      (unsigned)ksplit, mw, mh, a, ksplit);
}

cudaError_t read_front_faults(uint32_t *flags, bool clear)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return e;
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_front_faults, sizeof v);
    if (e != cudaSuccess)
        return e;
    *flags = v;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_front_faults, &zero, sizeof zero);
    }
    return e;
}

}  // namespace rc
