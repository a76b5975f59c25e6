// K3: K-norm, GPT-J RoPE and the paged insert of K and V.
//
// Page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.context",
// _ContextKvStoreKernel / _sum_squares_64 / _rope: one warp per (row, layer),
// lane j holding the GPT-J pair (2j, 2j+1) of every head, the head's sum of
// squares folded as even squares and odd squares separately by an xor
// butterfly, then even + odd; the normed key rounded to bf16; the rotation
// (fma(x, c, -(y*s)), fma(y, c, x*s)); K and V written as 4-byte words, so
// each warp store covers 128 contiguous bytes of one head.
//
// Differences from the pages' kernel: 8 warps (rows) per CTA instead of one;
// a slot past the cache or a position past the table skips the row and counts
// it in the caller's error word instead of writing out of bounds.
#include "rc_internal.cuh"

namespace rc {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void count_skip(int32_t *err, int lane) {
    if (err != nullptr && lane == 0)
        atomicAdd(err, 1);
}

// Writes one row's H heads of K' and V into its cache slot (lane = pair).
template <int H>
__device__ __forceinline__ void insert_row(uint16_t *cache, int64_t slot, int32_t block_size,
                                           const uint32_t (&ko)[H], const uint32_t (&vw)[H],
                                           int lane) {
    // Slots of a cache fit 32 bits (checked on the host).
    const uint32_t bs = (uint32_t)block_size;
    const uint32_t blk = (uint32_t)slot / bs;
    const uint32_t page = (uint32_t)slot - blk * bs;
    uint32_t *dst = reinterpret_cast<uint32_t *>(cache) + (((int64_t)blk * H) * bs + page) * kHeadDim + lane;
    const int64_t head_stride = (int64_t)bs * kHeadDim;      // in 4-byte words
#pragma unroll
    for (int h = 0; h < H; ++h) {
        dst[h * head_stride] = ko[h];
        dst[h * head_stride + kHeadDim / 2] = vw[h];          // V follows K
    }
}

template <int H, bool kRope>
__global__ void __launch_bounds__(kWarps * 32)
k3_kv_store(const __grid_constant__ StoreLaunch p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
    const int layer = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    if (row >= p.rows[layer])
        return;
    const int64_t *slots = p.slots[layer];
    if (slots == nullptr)
        return;
    // Every load first, as the pages' kernel does: the slot, the position and
    // the row's K and V words are independent, so their latencies overlap; a
    // skipped row wastes its K/V reads but never writes.
    const int64_t slot = __ldg(slots + row);
    const int64_t pos = kRope ? __ldg(p.positions + row) : 0;
    const uint32_t *kr = reinterpret_cast<const uint32_t *>(
        p.k + (int64_t)layer * p.k_layer_stride + row * p.k_row_stride) + lane;
    const uint32_t *vr = reinterpret_cast<const uint32_t *>(
        p.v + (int64_t)layer * p.v_layer_stride + row * p.v_row_stride) + lane;
    uint32_t kw[H], vw[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        kw[h] = __ldcs(kr + h * (kHeadDim / 2));
        vw[h] = __ldcs(vr + h * (kHeadDim / 2));
    }
    if (slot < 0)
        return;
    if (slot >= p.capacity || (kRope && (pos < 0 || pos >= p.max_position))) {
        count_skip(p.err, lane);
        return;
    }
    float c = 1.0f, s = 0.0f;
    if (kRope) {
        const unsigned short *cs = reinterpret_cast<const unsigned short *>(p.cos_sin) + pos * kHeadDim;
        c = __uint_as_float((uint32_t)__ldg(cs + lane) << 16);
        s = __uint_as_float((uint32_t)__ldg(cs + kHeadDim / 2 + lane) << 16);
    }

    uint32_t ko[H];
#pragma unroll
    for (int h = 0; h < H; ++h)
        ko[h] = knorm_rope_lane<kRope>(bf16_lo(kw[h]), bf16_hi(kw[h]), c, s, p.eps);
    insert_row<H>(p.caches[layer], slot, p.block_size, ko, vw, lane);
}

// The same store with one thread per key head.  A warp takes the 32 (row,
// head) keys of 32 / H consecutive rows of one layer: it copies their K and
// V into shared memory with coalesced 16-byte asynchronous copies (all in
// flight at once, no registers held), each lane then reads one whole key
// head (64 bf16), folds its sum of squares in registers in the butterfly's
// order (knorm_rope_head: the same bits as the lane version, without
// shuffles, and the square root and divide done once per head instead of
// once per lane), and K' and V leave for the cache with 16-byte stores, 8
// lanes per 128-byte half row.  Needs k, v and the caches 16-byte aligned
// and row / layer strides in multiples of 8 elements.
//
// Shared memory per warp: K and V of 32 heads, 8 chunks of 16 bytes each
// (logical chunk c of head e sits at chunk c ^ (e % 8), so the row-wise fill
// and the head-wise read are both free of bank conflicts), and with RoPE the
// 128-byte table rows of the warp's rows.
constexpr int kHeadsWarps = 4;

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *src, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}

template <int H, bool kRope>
__global__ void __launch_bounds__(kHeadsWarps * 32)
k3_kv_store_heads(const __grid_constant__ StoreLaunch p)
{
    constexpr int R = 32 / H;                     // rows per warp
    __shared__ uint4 ktile[kHeadsWarps][32][8];
    __shared__ uint4 vtile[kHeadsWarps][32][8];
    __shared__ uint4 cstile[kHeadsWarps][kRope ? R : 1][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int layer = blockIdx.y;
    const int64_t row0 = ((int64_t)blockIdx.x * kHeadsWarps + warp) * R;
    pdl_trigger();
    pdl_wait();
    const int64_t nrows = p.rows[layer];
    const int64_t *slots = p.slots[layer];
    if (slots == nullptr || row0 >= nrows)
        return;
    // chunk i of this lane: key e = 4 i + lane / 8 (row e / H, head e % H),
    // 16-byte piece lane % 8 of its 64 elements; rows past the layer's count
    // are zero-filled without a read
    const int piece = lane & 7;
    const uint16_t *kl = p.k + (int64_t)layer * p.k_layer_stride;
    const uint16_t *vl = p.v + (int64_t)layer * p.v_layer_stride;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = 4 * i + (lane >> 3);
        const int64_t row = row0 + e / H;
        const bool live = row < nrows;
        const int64_t r = live ? row : row0;
        const int h = e % H;
        cp_async16(&ktile[warp][e][piece ^ (e & 7)], kl + r * p.k_row_stride + h * kHeadDim + 8 * piece, live);
        cp_async16(&vtile[warp][e][piece ^ (e & 7)], vl + r * p.v_row_stride + h * kHeadDim + 8 * piece, live);
    }
    // this lane's key: row row0 + lane / H, head lane % H
    const int64_t my_row = row0 + lane / H;
    int64_t slot = -1, pos = 0;
    if (my_row < nrows) {
        slot = __ldg(slots + my_row);
        if (kRope)
            pos = __ldg(p.positions + my_row);
    }
    bool ok = slot >= 0;
    if (ok && (slot >= p.capacity || (kRope && (pos < 0 || pos >= p.max_position)))) {
        if (lane % H == 0)                        // counted once per (row, layer)
            count_skip(p.err, 0);
        ok = false;
    }
    if (kRope) {
        // table row of warp row r: logical chunk c in cstile[r][c ^ (r % 8)];
        // the lane of head 0 of each row hands its position to the copiers
        const int64_t tpos = ok ? pos : 0;
#pragma unroll
        for (int i = 0; i < (R * 8 + 31) / 32; ++i) {
            const int c = 32 * i + lane;
            const int r = c >> 3;
            const int64_t rp = __shfl_sync(0xFFFFFFFFu, tpos, (r * H) & 31);
            if (c < R * 8)
                cp_async16(&cstile[warp][r][(c ^ r) & 7], p.cos_sin + rp * kHeadDim + 8 * (c & 7), true);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    int64_t dst = -1;                             // the key's cache row (element offset)
    if (ok) {
        // Slots of a cache fit 32 bits (checked on the host).
        const uint32_t bs = (uint32_t)p.block_size;
        const uint32_t blk = (uint32_t)slot / bs;
        const uint32_t page = (uint32_t)slot - blk * bs;
        dst = (((int64_t)blk * H + lane % H) * bs + page) * (2 * kHeadDim);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
    uint16_t *cache = p.caches[layer];
    // V (a bit copy) leaves first
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = 4 * i + (lane >> 3);
        const int64_t d = __shfl_sync(0xFFFFFFFFu, dst, e);
        if (d >= 0)
            reinterpret_cast<uint4 *>(cache + d + kHeadDim)[piece] = vtile[warp][e][piece ^ (e & 7)];
    }
    __syncwarp();                                 // keeps V's registers apart from the head's
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 q = ktile[warp][lane][j ^ (lane & 7)];
        w[4 * j] = q.x; w[4 * j + 1] = q.y; w[4 * j + 2] = q.z; w[4 * j + 3] = q.w;
    }
    knorm_rope_head<kRope>(w, cstile[warp][kRope ? lane / H : 0], (lane / H) & 7, p.eps);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        ktile[warp][lane][j ^ (lane & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = 4 * i + (lane >> 3);
        const int64_t d = __shfl_sync(0xFFFFFFFFu, dst, e);
        if (d >= 0)
            reinterpret_cast<uint4 *>(cache + d)[piece] = ktile[warp][e][piece ^ (e & 7)];
    }
}

// Split-K projection finished and stored in one pass: the FP32 partials
// [splits, L, T, 128 H] are added in split order and rounded to bf16 (the
// same additions as the projection's reduce kernel), optionally written to
// kv_out, and stored like k3_kv_store.  One warp per (row, layer), 4 warps
// per CTA, so a whole workload's rows are resident in about one wave; lane
// j holds pair (2j, 2j+1) of each head.  Heads go in groups of kRsHeads,
// and the partials of up to kRsSplits splits of a group (K and V) are all in
// flight before the first add; the adds stay in split order.
constexpr int kRsWarps = 4;
constexpr int kRsHeads = 8;
constexpr int kRsSplits = 3;

template <bool kRope>
__global__ void __launch_bounds__(kRsWarps * 32, 3)
k3_reduce_store(const __grid_constant__ FusedStore fs, const float *__restrict__ partial,
                int32_t splits, int32_t L, int32_t T)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kRsWarps + warp;
    const int layer = blockIdx.y;
    const int H = fs.H;
    const int N = 2 * H * kHeadDim;
    pdl_trigger();
    pdl_wait();
    if (row >= T)
        return;
    const int64_t *slots = fs.slots[layer];
    const bool store = slots != nullptr && row < fs.rows[layer];
    int64_t slot = -1, pos = 0;
    if (store) {
        slot = __ldg(slots + row);
        if (kRope)
            pos = __ldg(fs.positions + row);
    }
    const int64_t plane = (int64_t)L * T * N;
    const float *prow = partial + ((int64_t)layer * T + row) * N + 2 * lane;
    const bool in_range = store && slot >= 0 && slot < fs.capacity &&
                          (!kRope || (pos >= 0 && pos < fs.max_position));
    if (store && slot >= 0 && !in_range && lane == 0)   // once per (row, layer)
        count_skip(fs.err, 0);
    // the table row (row 0 for rows that are not stored)
    float c = 1.0f, s = 0.0f;
    if (kRope) {
        const unsigned short *cs = reinterpret_cast<const unsigned short *>(fs.cos_sin) +
                                   (in_range ? pos : 0) * kHeadDim;
        c = __uint_as_float((uint32_t)__ldg(cs + lane) << 16);
        s = __uint_as_float((uint32_t)__ldg(cs + kHeadDim / 2 + lane) << 16);
    }
    uint32_t *dst_row = nullptr;
    if (in_range) {
        // Slots of a cache fit 32 bits (checked on the host).
        const uint32_t bs = (uint32_t)fs.block_size;
        const uint32_t blk = (uint32_t)slot / bs;
        const uint32_t page = (uint32_t)slot - blk * bs;
        dst_row = reinterpret_cast<uint32_t *>(fs.caches[layer]) +
                  (((int64_t)blk * H) * bs + page) * kHeadDim + lane;
    }
    uint32_t *kvo = fs.kv_out ? reinterpret_cast<uint32_t *>(fs.kv_out + ((int64_t)layer * T + row) * N) + lane
                              : nullptr;
    for (int h0 = 0; h0 < H; h0 += kRsHeads) {
        const int nh = min(kRsHeads, H - h0);
        float2 ka[kRsHeads], va[kRsHeads];
        for (int sp = 0; sp < splits; sp += kRsSplits) {
            float2 a[kRsSplits][kRsHeads], b[kRsSplits][kRsHeads];
#pragma unroll
            for (int u = 0; u < kRsSplits; ++u) {
#pragma unroll
                for (int q = 0; q < kRsHeads; ++q) {
                    if (sp + u < splits && q < nh) {
                        const float *pk = prow + (sp + u) * plane + (h0 + q) * kHeadDim;
                        a[u][q] = __ldcs(reinterpret_cast<const float2 *>(pk));
                        b[u][q] = __ldcs(reinterpret_cast<const float2 *>(pk + H * kHeadDim));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kRsSplits; ++u) {
#pragma unroll
                for (int q = 0; q < kRsHeads; ++q) {
                    if (sp + u < splits && q < nh) {
                        if (sp + u == 0) {
                            ka[q] = a[u][q];
                            va[q] = b[u][q];
                        } else {
                            ka[q].x = __fadd_rn(ka[q].x, a[u][q].x);
                            ka[q].y = __fadd_rn(ka[q].y, a[u][q].y);
                            va[q].x = __fadd_rn(va[q].x, b[u][q].x);
                            va[q].y = __fadd_rn(va[q].y, b[u][q].y);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kRsHeads; ++q) {
            if (q < nh) {
                const int h = h0 + q;
                const uint32_t kw = pack_bf16x2(ka[q].x, ka[q].y), vw = pack_bf16x2(va[q].x, va[q].y);
                if (kvo) {
                    kvo[h * (kHeadDim / 2)] = kw;
                    kvo[(H + h) * (kHeadDim / 2)] = vw;
                }
                if (in_range) {
                    uint32_t *dst = dst_row + (int64_t)h * fs.block_size * kHeadDim;
                    dst[0] = knorm_rope_lane<kRope>(bf16_lo(kw), bf16_hi(kw), c, s, fs.eps);
                    dst[kHeadDim / 2] = vw;           // V follows K
                }
            }
        }
    }
}

// 16-byte access to K, V, the table and every cache of the chunk.
bool vector_ok(const StoreLaunch &p, int32_t layers) {
    const auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    if (!a16(p.k) || !a16(p.v) || (p.cos_sin && !a16(p.cos_sin)))
        return false;
    if ((p.k_layer_stride | p.k_row_stride | p.v_layer_stride | p.v_row_stride) & 7)
        return false;
    for (int32_t i = 0; i < layers; ++i)
        if (p.slots[i] && !a16(p.caches[i]))
            return false;
    return true;
}

template <int H>
cudaError_t launch_h(const StoreLaunch &p, int32_t layers, cudaStream_t stream) {
    const dim3 block(kWarps * 32);
    if (vector_ok(p, layers)) {
        constexpr int rows_per_cta = kHeadsWarps * (32 / H);
        const dim3 grid((unsigned)((p.grid_rows + rows_per_cta - 1) / rows_per_cta), (unsigned)layers);
        if (p.cos_sin)
            return launch_pdl(k3_kv_store_heads<H, true>, grid, dim3(kHeadsWarps * 32), 0, stream, 1, p);
        return launch_pdl(k3_kv_store_heads<H, false>, grid, dim3(kHeadsWarps * 32), 0, stream, 1, p);
    }
    const dim3 grid((unsigned)((p.grid_rows + kWarps - 1) / kWarps), (unsigned)layers);
    if (p.cos_sin)
        return launch_pdl(k3_kv_store<H, true>, grid, block, 0, stream, 1, p);
    return launch_pdl(k3_kv_store<H, false>, grid, block, 0, stream, 1, p);
}

}  // namespace

cudaError_t launch_reduce_store(const FusedStore &fs, const float *partial, int32_t splits,
                                int32_t L, int32_t T, cudaStream_t stream)
{
    const dim3 grid((unsigned)((T + kRsWarps - 1) / kRsWarps), (unsigned)L);
    if (fs.cos_sin)
        return launch_pdl(k3_reduce_store<true>, grid, dim3(kRsWarps * 32), 0, stream, 1, fs, partial,
                          splits, L, T);
    return launch_pdl(k3_reduce_store<false>, grid, dim3(kRsWarps * 32), 0, stream, 1, fs, partial,
                      splits, L, T);
}

cudaError_t launch_kv_store(const StoreLaunch &p, int32_t H, int32_t layers, cudaStream_t stream)
{
    switch (H) {
    case 1: return launch_h<1>(p, layers, stream);
    case 2: return launch_h<2>(p, layers, stream);
    case 4: return launch_h<4>(p, layers, stream);
    case 8: return launch_h<8>(p, layers, stream);
    case 16: return launch_h<16>(p, layers, stream);
    case 32: return launch_h<32>(p, layers, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rc
