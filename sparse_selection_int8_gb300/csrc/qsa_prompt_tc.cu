// qsa_prompt_tc.cu -- tensor-core path for prompt-shaped calls (step a6).
//
// The pages run a prompt chunk through the decode kernel ("Strata PR #2220,
// attn_chunk_q8_v3_kernel", prompt-shaped parity: 2,048 queries against 32K
// INT8 cells).  With thousands of query rows per KV head the two
// contractions are dense, so this path puts the query rows on the MMA's M
// dimension and streams the selected cells through it, flash-attention
// style:
//
//   staging   one pass resolves every listed cell through the page table
//             (a1) and writes tensor-core-ready images to the workspace:
//             K codes as 16-bit floats (exact), V as f16(code x v_scale),
//             per-cell k_scale*softmax_scale*log2(e), a 0/-inf mask bias and
//             the cell's logical position (read only by calls with causal
//             limits per query), and the queries, each 128-row or 128-cell
//             tile a contiguous 64 KB block in the 128-byte-swizzled layout;
//   main      one CTA per (128-row query tile, chunk) loads image tiles with
//             bulk async copies (a copy warp) and runs, per 128-cell tile,
//               S = Q . K_code^T        (M=128 rows, N=128 cells, K=256)
//               P = 2^(S*ksc + bias - m_ref)      (online softmax)
//               O += P . V_hat          (M=128 rows, N=256 d, K=128 cells)
//             with two S buffers and O in tensor memory, so the MMA warp
//             runs S of the next tile while the softmax warps work on this
//             one; P (f16) overwrites its own S in tensor memory and is the
//             A operand of P . V_hat there.  O is rescaled only when a
//             row's max grows by more than 2^8 over its reference, so P
//             stays below 256 and f16 holds it; the partial is brought to
//             the true running max at the end.
// The partials have the decode path's layout and go to the same merge.
// Calls with causal limits run a separate instantiation whose softmax also
// sets the scores of cells at or past the row's limit to -inf.
//
// Queries keep their own 16-bit type (bf16 queries with bf16 K codes; f32
// queries are rounded to f16 and use f16 K codes), since one tcgen05.mma
// takes A and B of the same type.  V_hat = f16(code * v_scale) needs
// |v_scale| * 127 < 65504.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qsa_internal.cuh"
#include "qsa_sm100.cuh"

namespace qsa {
namespace {

using namespace sm100;

constexpr int kTile = 128;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2; // 64 KB image tile

// Tensor-memory column of P's packed f16 pair k (cells 2k, 2k+1) inside its
// S buffer: the softmax thread of column half h holds S columns 64h..64h+63
// and writes its 32 pairs over the first half of them.
__device__ __forceinline__ uint32_t p_col(int k) { return (uint32_t)(k < 32 ? k : 32 + k); }

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    if (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ---------------------------------------------------------------- staging

// One CTA per 128-cell image tile of (chunk c, tile j) of one (sequence, KV
// head).  Cells past the chunk or the list are masked (zero rows, bias -inf).
template <bool QBF16>
__global__ void __launch_bounds__(256) qsa_prompt_stage_kv(const Params p, const PromptImages im)
{
    __shared__ int s_slot[kTile];
    __shared__ float s_vs[kTile];
    const int tile = blockIdx.x;
    const int g = blockIdx.y, b = blockIdx.z;
    const int c = tile / im.tiles_per_chunk, j = tile % im.tiles_per_chunk;
    int start, n;
    seq_range(p, b, &start, &n);
    const size_t kv_base = ((size_t)b * p.G + g) * p.pool_cells;
    const size_t tile_id = (((size_t)b * p.G + g) * p.n_chunks + c) * im.tiles_per_chunk + j;
    const long long c0 = (long long)c * p.chunk_cells;
    const long long lo = c0 + (long long)j * kTile;
    const long long hi = min(min(c0 + p.chunk_cells, (long long)n), lo + kTile);
    const int tid = threadIdx.x;
    if (tid < kTile) {
        int slot = -1, pos = INT_MAX;
        if (lo + tid < hi) {
            pos = __ldg(p.sel + start + lo + tid);
            slot = resolve_slot(p, b, pos);
        }
        im.pos[tile_id * kTile + tid] = pos;
        s_slot[tid] = slot;
        s_vs[tid] = slot >= 0 ? __ldg(p.v_scale + kv_base + slot) : 0.f;
        im.ksc[tile_id * kTile + tid] = slot >= 0 ? __ldg(p.k_scale + kv_base + slot) * p.scale_log2 : 0.f;
        im.bias[tile_id * kTile + tid] = slot >= 0 ? 0.f : -INFINITY;
    }
    __syncthreads();
    uint8_t *kimg = static_cast<uint8_t *>(im.k) + tile_id * kTileBytes;
    uint8_t *vimg = static_cast<uint8_t *>(im.v) + tile_id * kTileBytes;
    for (int e = tid; e < kTile * 16; e += blockDim.x) {
        const int cell = e >> 4, piece = e & 15; // 16 codes = d 16*piece .. +15
        const int slot = s_slot[cell];
        uint4 kr = make_uint4(0, 0, 0, 0), vr = make_uint4(0, 0, 0, 0);
        if (slot >= 0) {
            kr = ldg_nc_v4(p.k_pool + (kv_base + slot) * kHeadDim + piece * 16);
            vr = ldg_nc_v4(p.v_pool + (kv_base + slot) * kHeadDim + piece * 16);
        }
        const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w}, vw[4] = {vr.x, vr.y, vr.z, vr.w};
        const float vsc = s_vs[cell];
        uint32_t ko[8], vo[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float k0 = (float)(int8_t)(kw[q] & 0xff), k1 = (float)(int8_t)((kw[q] >> 8) & 0xff);
            const float k2 = (float)(int8_t)((kw[q] >> 16) & 0xff), k3 = (float)(int8_t)(kw[q] >> 24);
            ko[2 * q] = pack2<QBF16>(k0, k1);
            ko[2 * q + 1] = pack2<QBF16>(k2, k3);
            const float v0 = (float)(int8_t)(vw[q] & 0xff) * vsc, v1 = (float)(int8_t)((vw[q] >> 8) & 0xff) * vsc;
            const float v2 = (float)(int8_t)((vw[q] >> 16) & 0xff) * vsc, v3 = (float)(int8_t)(vw[q] >> 24) * vsc;
            vo[2 * q] = pack2<false>(v0, v1);
            vo[2 * q + 1] = pack2<false>(v2, v3);
        }
        const uint32_t off0 = kmajor_sw128_off(cell, piece * 16, kTile);
        const uint32_t off1 = kmajor_sw128_off(cell, piece * 16 + 8, kTile);
        *reinterpret_cast<uint4 *>(kimg + off0) = make_uint4(ko[0], ko[1], ko[2], ko[3]);
        *reinterpret_cast<uint4 *>(kimg + off1) = make_uint4(ko[4], ko[5], ko[6], ko[7]);
        *reinterpret_cast<uint4 *>(vimg + off0) = make_uint4(vo[0], vo[1], vo[2], vo[3]);
        *reinterpret_cast<uint4 *>(vimg + off1) = make_uint4(vo[4], vo[5], vo[6], vo[7]);
    }
}

// One CTA per 128-row query tile of one (sequence, KV head); row r = t*H + j.
template <bool QBF16>
__global__ void __launch_bounds__(256) qsa_prompt_stage_q(const Params p, const PromptImages im)
{
    const int mt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    uint8_t *qimg = static_cast<uint8_t *>(im.q) + (((size_t)b * p.G + g) * im.row_tiles + mt) * kTileBytes;
    const int GH = p.G * p.H;
    for (int e = threadIdx.x; e < kTile * 32; e += blockDim.x) {
        const int row = e >> 5, piece = e & 31; // 8 values = d 8*piece .. +7
        const int r = mt * kTile + row;
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (r < p.R) {
            const int t = r / p.H, j = r % p.H;
            const size_t off = (((size_t)b * p.T + t) * GH + (size_t)g * p.H + j) * kHeadDim + piece * 8;
            if (p.q_bf16) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) + off);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    f[2 * q] = bf16_bits_to_f32(w[q] & 0xffff);
                    f[2 * q + 1] = bf16_bits_to_f32(w[q] >> 16);
                }
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(p.q) + off);
                const float4 x = src[0], y = src[1];
                f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
                f[4] = y.x; f[5] = y.y; f[6] = y.z; f[7] = y.w;
            }
        }
        const uint4 v = make_uint4(pack2<QBF16>(f[0], f[1]), pack2<QBF16>(f[2], f[3]),
                                   pack2<QBF16>(f[4], f[5]), pack2<QBF16>(f[6], f[7]));
        *reinterpret_cast<uint4 *>(qimg + kmajor_sw128_off(row, piece * 8, kTile)) = v;
    }
}

// ---------------------------------------------------------------- main

constexpr int kSoftThreads = 2 * kTile;       // two threads per query row (column halves)
constexpr int kMmaWarp = kSoftThreads / 32;   // 8: issues the MMAs (one thread)
constexpr int kLoadWarp = kMmaWarp + 1;       // 9: bulk copies of Q, K and the score factors (one thread)
constexpr int kVLoadWarp = kLoadWarp + 1;     // 10: bulk copies of V (one thread)
constexpr int kThreads = kSoftThreads + 96;   // 352
constexpr uint32_t kBarSoft = 1;              // named barrier of the softmax warps
constexpr long long kDrainCycles = 1ll << 30; // bound of the waits before the CTA leaves

// (Shared memory holds the Q, K and V tiles and this.)
struct PromptSmem {
    float ksc[kTile];           // per-cell score factors of the current tile
    float bias[kTile];          // 0 or -inf (masked cell)
    int32_t pos[kTile];         // the cells' logical positions (calls with causal limits)
    float rowmax[2][kTile];     // [column half][row]; the rows' sums at the end
    uint64_t bar_q, k_full, k_empty, v_full, o_done, p_full, c_full, mma_done;
    uint64_t s_full[2], s_empty[2];
    uint32_t tmem;
    int32_t abort;
};
static_assert(sizeof(PromptSmem) <= 3072, "shared memory of the prompt kernel");

__device__ __forceinline__ bool wait_bar(const Params &p, PromptSmem &ms, uint64_t *bar, uint32_t parity)
{
    if (ms.abort) return false;
    if (!mbar_wait(bar, parity, p.wait_cycles)) {
        atomicExch(&ms.abort, 1);
        raise_status(p, QSA_STATUS_TIMEOUT);
        return false;
    }
    return true;
}

// Warp roles: softmax warps 0-7 (warp w owns query rows 32*(w%4)..+31, its
// TMEM lanes, and column half w/4 of S (cells) and of O (dimensions)); MMA
// warp 8; bulk-copy warp 9.  Two S buffers in tensor memory let S of tile
// j+1 run on the tensor cores while the softmax works on tile j; the
// tensor pipe then takes O += P.V of tile j, with P of tile j in tensor
// memory where S of tile j was.  S of tile j+2 reuses that buffer; it is
// issued after P.V of tile j by the same thread, and the tensor pipe runs
// one thread's MMAs in order.  K and V have one shared-memory buffer each
// (with Q resident, shared memory holds no more): K of tile j+1 is copied
// as soon as S of tile j is done (during P.V of tile j-1), V of tile j+1 as
// soon as P.V of tile j is done (during S of tile j+2), the score factors
// once the softmax has read the previous ones.
template <bool QBF16, bool LIM>
__global__ void __launch_bounds__(kThreads, 1) qsa_prompt_tc_kernel(const Params p, const PromptImages im)
{
    // The operand tiles need 1024-byte alignment (128-byte swizzle atoms);
    // the dynamic shared memory of a kernel without static shared memory
    // starts there.  The check keeps a misplaced window from being used.
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) raise_status(p, QSA_STATUS_LAUNCH);
        return;
    }
    const uint32_t s_q = smem_u32(smem), s_k = s_q + kTileBytes, s_v = s_k + kTileBytes;
    PromptSmem &ms = *reinterpret_cast<PromptSmem *>(smem + 3 * kTileBytes);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x / p.n_chunks, c = blockIdx.x % p.n_chunks;
    const int g = blockIdx.y, b = blockIdx.z;
    int start, n;
    seq_range(p, b, &start, &n);
    cudaTriggerProgrammaticLaunchCompletion();
    if ((long long)c * p.chunk_cells >= n) return; // no such chunk: the merge skips it
    const int cells = (int)min((long long)p.chunk_cells, (long long)n - (long long)c * p.chunk_cells);
    const int n_tiles = (cells + kTile - 1) / kTile;
    const size_t tile0 = (((size_t)b * p.G + g) * p.n_chunks + c) * im.tiles_per_chunk;
    const uint8_t *kimg = static_cast<const uint8_t *>(im.k) + tile0 * kTileBytes;
    const uint8_t *vimg = static_cast<const uint8_t *>(im.v) + tile0 * kTileBytes;
    const uint8_t *qimg = static_cast<const uint8_t *>(im.q) + (((size_t)b * p.G + g) * im.row_tiles + mt) * kTileBytes;
    const float *kscg = im.ksc + tile0 * kTile, *biasg = im.bias + tile0 * kTile;
    const int32_t *posg = im.pos + tile0 * kTile;

    if (tid == 0) {
        mbar_init(&ms.bar_q, 1);
        mbar_init(&ms.k_full, 1);
        mbar_init(&ms.k_empty, 1);
        mbar_init(&ms.v_full, 1);
        mbar_init(&ms.o_done, 1);
        mbar_init(&ms.p_full, kSoftThreads);
        mbar_init(&ms.c_full, 1);
        mbar_init(&ms.mma_done, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.s_empty[i], kSoftThreads);
        }
        ms.abort = 0;
        fence_mbar_init();
    }
    if (w == 0) {
        tmem_alloc(&ms.tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem, t_o = tmem + 2 * kTile; // S buffers at columns 0 and 128

    if (w == kLoadWarp) {
        // ================================================================ bulk copies (Q, K, factors)
        // K and V have their own copy threads: the tensor pipe frees the K
        // buffer (S of a tile) before the V buffer (P.V of the previous
        // tile), and neither copy waits for the other's buffer.
        if (lane == 0) {
            auto load_k = [&](int j) {
                mbar_arrive_expect_tx(&ms.k_full, kTileBytes);
                bulk_g2s(smem + kTileBytes, kimg + (size_t)j * kTileBytes, kTileBytes, &ms.k_full);
            };
            auto load_c = [&](int j) {
                mbar_arrive_expect_tx(&ms.c_full, (LIM ? 3 : 2) * kTile * 4);
                bulk_g2s(ms.ksc, kscg + (size_t)j * kTile, kTile * 4, &ms.c_full);
                bulk_g2s(ms.bias, biasg + (size_t)j * kTile, kTile * 4, &ms.c_full);
                if (LIM) bulk_g2s(ms.pos, posg + (size_t)j * kTile, kTile * 4, &ms.c_full);
            };
            mbar_arrive_expect_tx(&ms.bar_q, kTileBytes);
            bulk_g2s(smem, qimg, kTileBytes, &ms.bar_q);
            load_k(0);
            load_c(0);
            int nk = 1, nc = 1; // copies issued
            for (int j = 0; j + 1 < n_tiles && !ms.abort; ++j) {
                // K of tile j+1 once S of tile j is done
                if (!wait_bar(p, ms, &ms.k_empty, (uint32_t)j & 1u)) break;
                load_k(j + 1);
                ++nk;
                // score factors of tile j+1 once the softmax of tile j has read its own
                if (!wait_bar(p, ms, &ms.s_empty[j & 1], (uint32_t)(j >> 1) & 1u)) break;
                load_c(j + 1);
                ++nc;
            }
            // before the CTA leaves (also after a time-out): every copy of
            // this thread landed.  The k-th copy on a barrier completes its
            // phase k - 1, and nothing else arrives on these barriers.
            mbar_wait(&ms.bar_q, 0, kDrainCycles);
            mbar_wait(&ms.k_full, (uint32_t)(nk - 1) & 1u, kDrainCycles);
            mbar_wait(&ms.c_full, (uint32_t)(nc - 1) & 1u, kDrainCycles);
        }
        __syncwarp();
    } else if (w == kVLoadWarp) {
        // ================================================================ bulk copies (V)
        if (lane == 0) {
            auto load_v = [&](int j) {
                mbar_arrive_expect_tx(&ms.v_full, kTileBytes);
                bulk_g2s(smem + 2 * kTileBytes, vimg + (size_t)j * kTileBytes, kTileBytes, &ms.v_full);
            };
            load_v(0);
            int nv = 1;
            for (int j = 0; j + 1 < n_tiles && !ms.abort; ++j) {
                // V of tile j+1 once P.V of tile j is done
                if (!wait_bar(p, ms, &ms.o_done, (uint32_t)j & 1u)) break;
                load_v(j + 1);
                ++nv;
            }
            mbar_wait(&ms.v_full, (uint32_t)(nv - 1) & 1u, kDrainCycles); // every copy landed
        }
        __syncwarp();
    } else if (w == kMmaWarp) {
        // ================================================================ MMA issue
        if (lane == 0) {
            const uint32_t idesc_s = idesc_f16(kTile, kTile, QBF16, QBF16, false, false);
            const uint32_t idesc_o = idesc_f16(kTile, kHeadDim, false, false, false, true);
            auto issue_s = [&](int j) {
                const uint32_t t_s = tmem + (uint32_t)(j & 1) * kTile;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint64_t ad = smem_desc(s_q + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(s_k + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024);
                    mma_f16_ss(t_s, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&ms.k_empty);
                mma_commit(&ms.s_full[j & 1]);
            };
            wait_bar(p, ms, &ms.bar_q, 0);
            wait_bar(p, ms, &ms.k_full, 0);
            tc_fence_after();
            issue_s(0);
            for (int j = 0; j < n_tiles && !ms.abort; ++j) {
                if (j + 1 < n_tiles) {
                    wait_bar(p, ms, &ms.k_full, (uint32_t)(j + 1) & 1u);
                    if (j >= 1) wait_bar(p, ms, &ms.s_empty[(j + 1) & 1], (uint32_t)((j - 1) >> 1) & 1u);
                    tc_fence_after();
                    issue_s(j + 1);
                }
                wait_bar(p, ms, &ms.p_full, (uint32_t)j & 1u);
                wait_bar(p, ms, &ms.v_full, (uint32_t)j & 1u);
                tc_fence_after();
                const uint32_t t_p = tmem + (uint32_t)(j & 1) * kTile; // P of tile j
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint64_t bd = smem_desc(s_v + kk * 2048, kTile * 128, 1024);
                    mma_f16_ts(t_o, t_p + p_col(8 * kk), bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&ms.o_done);
            }
            // before the CTA leaves (also after a time-out): every MMA of this
            // thread complete, so tensor memory is idle when it is freed
            mma_commit(&ms.mma_done);
            mbar_wait(&ms.mma_done, 0, kDrainCycles);
        }
        __syncwarp();
    } else {
        // ================================================================ softmax
        const int row = 32 * (w & 3) + lane, hc = w >> 2;
        const uint32_t t_lane = (uint32_t)(32 * (w & 3)) << 16;
        float m_run = -INFINITY, m_ref = -INFINITY, l = 0.f;
        int lim = INT_MAX; // causal limit of this row's query: it sees positions below it
        if (LIM && mt * kTile + row < p.R)
            lim = __ldg(p.q_limit + (size_t)b * p.T + (mt * kTile + row) / p.H);
        for (int j = 0; j < n_tiles; ++j) {
            const int par = j & 1;
            wait_bar(p, ms, &ms.c_full, (uint32_t)j & 1u);
            wait_bar(p, ms, &ms.s_full[par], (uint32_t)(j >> 1) & 1u);
            tc_fence_after();
            // ---- this thread's 64 scaled, masked scores and the row max
            float sv[64];
#pragma unroll
            for (int c16 = 0; c16 < 4; ++c16)
                tmem_ld16(tmem + (uint32_t)par * kTile + t_lane + hc * 64 + c16 * 16, sv + c16 * 16);
            tmem_wait_ld();
            regs_after_wait<64>(sv);
            float mx = -INFINITY;
#pragma unroll
            for (int i4 = 0; i4 < 16; ++i4) { // the factors by 16-byte broadcast loads
                const float4 kf = *reinterpret_cast<const float4 *>(&ms.ksc[hc * 64 + 4 * i4]);
                const float4 bf = *reinterpret_cast<const float4 *>(&ms.bias[hc * 64 + 4 * i4]);
                sv[4 * i4] = fmaf(sv[4 * i4], kf.x, bf.x);
                sv[4 * i4 + 1] = fmaf(sv[4 * i4 + 1], kf.y, bf.y);
                sv[4 * i4 + 2] = fmaf(sv[4 * i4 + 2], kf.z, bf.z);
                sv[4 * i4 + 3] = fmaf(sv[4 * i4 + 3], kf.w, bf.w);
                if (LIM) {
                    const int4 pf = *reinterpret_cast<const int4 *>(&ms.pos[hc * 64 + 4 * i4]);
                    if (pf.x >= lim) sv[4 * i4] = -INFINITY;
                    if (pf.y >= lim) sv[4 * i4 + 1] = -INFINITY;
                    if (pf.z >= lim) sv[4 * i4 + 2] = -INFINITY;
                    if (pf.w >= lim) sv[4 * i4 + 3] = -INFINITY;
                }
                mx = fmaxf(mx, fmaxf(fmaxf(sv[4 * i4], sv[4 * i4 + 1]), fmaxf(sv[4 * i4 + 2], sv[4 * i4 + 3])));
            }
            tc_fence_before();
            mbar_arrive(&ms.s_empty[par]); // S buffer of this parity and the score factors free
            // every softmax thread has read the previous tile's row maxima
            // once P of that tile is complete
            if (j >= 1) wait_bar(p, ms, &ms.p_full, (uint32_t)(j - 1) & 1u);
            ms.rowmax[hc][row] = mx;
            named_bar(kBarSoft, kSoftThreads);
            mx = fmaxf(ms.rowmax[0][row], ms.rowmax[1][row]);
            // rescale O (and l) when this row's max outgrows its reference by 2^8
            bool rescale = false;
            float factor = 1.f;
            if (mx > -INFINITY) {
                if (m_ref == -INFINITY) {
                    m_ref = mx;
                } else if (mx > m_ref + 8.f) {
                    factor = fast_exp2(m_ref - mx);
                    l *= factor;
                    m_ref = mx;
                    rescale = true;
                }
                m_run = fmaxf(m_run, mx);
            }
            // P of this tile into registers first (the exponentials overlap P.V
            // of tile j-1 on the tensor cores); a row with no valid cell yet
            // keeps m_ref = -inf and only -inf scores: subtract 0 instead, so
            // they give 2^-inf = 0, not NaN
            const float m_sub = m_ref > -INFINITY ? m_ref : 0.f;
            float lp[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t hw[32];
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
                const float p0 = fast_exp2(sv[i] - m_sub);
                const float p1 = fast_exp2(sv[i + 1] - m_sub);
                lp[(i >> 1) & 3] += p0 + p1;
                hw[i >> 1] = pack2<false>(p0, p1);
            }
            // P over this thread's half of S (already in registers)
            const uint32_t t_p = tmem + (uint32_t)par * kTile + t_lane + hc * 64;
            tmem_st16u(t_p, hw);
            tmem_st16u(t_p + 16, hw + 16);
            if (__any_sync(0xffffffffu, rescale)) {
                // O is rescaled in place once P.V of tile j-1 is done (S of
                // tile j, done, was issued after P.V of tile j-2, so the
                // barrier is at most one phase behind)
                if (j >= 1) wait_bar(p, ms, &ms.o_done, (uint32_t)(j - 1) & 1u);
                tc_fence_after();
#pragma unroll 1
                for (int c16 = 0; c16 < 8; ++c16) {
                    float ov[16];
                    tmem_ld16(t_o + t_lane + hc * 128 + c16 * 16, ov);
                    tmem_wait_ld();
                    regs_after_wait<16>(ov);
#pragma unroll
                    for (int i = 0; i < 16; ++i) ov[i] *= factor;
                    tmem_st16(t_o + t_lane + hc * 128 + c16 * 16, ov);
                }
                tmem_wait_st();
            }
            l += (lp[0] + lp[1]) + (lp[2] + lp[3]);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&ms.p_full);
        }

        // ---- the partial relative to the row's true maximum.  The waits
        // test phase parity, so they go one phase at a time: S of the last
        // tile was issued after P.V of the tile three back, so the barrier
        // is at most two phases behind here.
        if (n_tiles >= 2) wait_bar(p, ms, &ms.o_done, (uint32_t)(n_tiles - 2) & 1u);
        wait_bar(p, ms, &ms.o_done, (uint32_t)(n_tiles - 1) & 1u); // last P.V done
        tc_fence_after();
        wait_bar(p, ms, &ms.p_full, (uint32_t)(n_tiles - 1) & 1u); // (row maxima read)
        ms.rowmax[hc][row] = l; // reused for the two halves' sums
        named_bar(kBarSoft, kSoftThreads);
        const int r = mt * kTile + row;
        const size_t base = (((size_t)b * p.G + g) * p.n_chunks + c) * p.R;
        const float fin = (m_run > -INFINITY && m_ref < m_run) ? fast_exp2(m_ref - m_run) : 1.f;
        if (r < p.R && hc == 0) {
            p.part_m[base + r] = m_run > -INFINITY ? m_run * kLn2 : -INFINITY;
            p.part_l[base + r] = m_run > -INFINITY ? (ms.rowmax[0][row] + ms.rowmax[1][row]) * fin : 0.f;
        }
#pragma unroll 1
        for (int c16 = 0; c16 < 8; ++c16) {
            float ov[16];
            tmem_ld16(t_o + t_lane + hc * 128 + c16 * 16, ov);
            tmem_wait_ld();
            regs_after_wait<16>(ov);
            if (r < p.R) {
                float4 *dst = reinterpret_cast<float4 *>(p.part_o + (base + r) * kHeadDim + hc * 128 + c16 * 16);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a0 = m_run > -INFINITY ? ov[4 * i] * fin : 0.f;
                    const float a1 = m_run > -INFINITY ? ov[4 * i + 1] * fin : 0.f;
                    const float a2 = m_run > -INFINITY ? ov[4 * i + 2] * fin : 0.f;
                    const float a3 = m_run > -INFINITY ? ov[4 * i + 3] * fin : 0.f;
                    dst[i] = make_float4(a0, a1, a2, a3);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == 0) tmem_dealloc(tmem, 512);
}

template <bool QBF16, bool LIM>
cudaError_t launch_prompt(const Params &p, const PromptImages &im, cudaStream_t stream)
{
    dim3 gkv((unsigned)(p.n_chunks * im.tiles_per_chunk), (unsigned)p.G, (unsigned)p.n_seq);
    qsa_prompt_stage_kv<QBF16><<<gkv, 256, 0, stream>>>(p, im);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 gq((unsigned)im.row_tiles, (unsigned)p.G, (unsigned)p.n_seq);
    qsa_prompt_stage_q<QBF16><<<gq, 256, 0, stream>>>(p, im);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int bytes = (int)(3 * kTileBytes + sizeof(PromptSmem));
    if ((e = cudaFuncSetAttribute(qsa_prompt_tc_kernel<QBF16, LIM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  bytes)) != cudaSuccess)
        return e;
    dim3 gm((unsigned)(im.row_tiles * p.n_chunks), (unsigned)p.G, (unsigned)p.n_seq);
    qsa_prompt_tc_kernel<QBF16, LIM><<<gm, kThreads, bytes, stream>>>(p, im);
    return cudaGetLastError();
}

} // namespace

size_t prompt_image_bytes(int n_seq, int G, int R, int chunk_cells, int n_chunks, size_t *k_bytes,
                          size_t *q_bytes, size_t *cell_bytes)
{
    const size_t tpc = ((size_t)chunk_cells + kTile - 1) / kTile;
    const size_t row_tiles = ((size_t)R + kTile - 1) / kTile;
    *k_bytes = (size_t)n_seq * G * n_chunks * tpc * kTileBytes;
    *q_bytes = (size_t)n_seq * G * row_tiles * kTileBytes;
    *cell_bytes = (size_t)n_seq * G * n_chunks * tpc * kTile * sizeof(float);
    return 2 * *k_bytes + *q_bytes + 3 * *cell_bytes;
}

cudaError_t launch_prompt_tc(const Params &p, const PromptImages &im, cudaStream_t stream)
{
    if (p.n_chunks == 0) return cudaSuccess;
    if (p.q_limit)
        return p.q_bf16 ? launch_prompt<true, true>(p, im, stream) : launch_prompt<false, true>(p, im, stream);
    return p.q_bf16 ? launch_prompt<true, false>(p, im, stream) : launch_prompt<false, false>(p, im, stream);
}

} // namespace qsa
