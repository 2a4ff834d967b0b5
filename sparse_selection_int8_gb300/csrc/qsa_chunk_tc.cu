// qsa_chunk_tc.cu -- tensor-core chunk kernel for decode windows (steps a1-a4).
//
// What it computes is the chunk step of "Strata PR #2220,
// attn_chunk_q8_v3_kernel": each chunk of the selected list yields partials
// (max m, sum of exponentials l, unnormalised P.V o) for every query row
// (T queries x H heads of one KV head).  The pages' Turing kernel reads each
// cell once for all 12 heads and does the dot products with warp shuffles;
// here both contractions run on the 5th-generation tensor cores with the
// cells on the MMA's M dimension, because a decode window has only 12-64
// query rows:
//
//   S^T[cell][row] = K_hat[cell][:] . Q[row][:]       M=128 cells, N=rows, K=256
//   O^T[d][row]    = V_hat^T[d][cell] . P^T[cell][row] M=128 d (x2), N=rows, K=128 cells
//
// INT8 codes convert exactly to f16 (|code| <= 127); the K scale multiplies
// the fp32 score after the MMA, and the V scale (divided by the group's
// largest V scale, so P stays in [0, 1]) multiplies P before it is rounded
// to f16; the group's largest scale multiplies the fp32 result.  Queries are
// rounded to f16.  Accumulation is fp32 in tensor memory.
//
// CTA = 1 producer warp + 8 consumer warps, persistent over a contiguous
// range of non-empty (sequence, KV head, chunk) items:
//   producer  resolves list entry -> page slot (a1) and streams the cells' K
//             and V rows (256 B each) with bulk async copies into a ring of
//             raw stages, plus the two per-cell scales with 4-byte cp.async;
//   consumers dequantise a stage into an f16 tile in the tensor cores'
//             128-byte-swizzled layout, issue tcgen05.mma from one thread,
//             and run the softmax (max via redux, sum via a reduce-scatter
//             butterfly), all in a fixed order, so partials are bit-identical
//             run to run.
// A chunk is processed in groups of up to 256 cells (two M tiles) that share
// one max; longer chunks combine their groups in registers.
//
// Every wait is bounded; a wait that runs out raises QSA_STATUS_TIMEOUT and
// the kernel runs to its end without further waiting.
#include <cuda_fp16.h>

#include "qsa_internal.cuh"
#include "qsa_sm100.cuh"

namespace qsa {
namespace {

using namespace sm100;

constexpr int kTile = 128;          // cells per MMA tile (M)
constexpr int kMaxTiles = 2;        // tiles per softmax group
constexpr int kGroupCells = kTile * kMaxTiles;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr uint32_t kOddRows = 64 * 256 + 64;        // odd rows start 64 B past a 128-B line
constexpr uint32_t kStageRowBytes = kOddRows + 64 * 256;
constexpr uint32_t kStageSlots = kStageRowBytes;     // int32[128]
constexpr uint32_t kStageKs = kStageSlots + 512;     // f32[128]
constexpr uint32_t kStageVs = kStageKs + 512;        // f32[128]
constexpr uint32_t kStageBytes = ((kStageVs + 512) + 127) / 128 * 128;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTileF16Bytes = kTile * kHeadDim * 2; // 64 KB

struct Layout {
    uint32_t off_kv, off_q, off_p, off_raw, n_stages, off_misc, total;
};

// Misc area: per-group cell info, reduction scratch, per-row values, barriers.
struct Misc {
    int32_t cell_slot[kMaxTiles][kTile];
    float cell_ks[kMaxTiles][kTile];
    float cell_vs[kMaxTiles][kTile];
    float red_max[2][4][32];
    float red_sum[2][4][32];
    float red_vs[2][4];
    float row_fa[64], row_fb[64], row_m[64], row_l[64], row_mrun[64], row_lrun[64];
    float sigma;
    int32_t abort;
    uint32_t tmem;
    uint64_t full[4], empty[4], mma;
};

__host__ __device__ inline Layout make_layout(int N, int n_stages)
{
    Layout L;
    L.off_kv = 0;
    L.off_q = kTileF16Bytes;
    L.off_p = L.off_q + (uint32_t)N * kHeadDim * 2;
    L.off_raw = L.off_p + (uint32_t)kMaxTiles * N * kTile * 2;
    L.n_stages = (uint32_t)n_stages;
    L.off_misc = L.off_raw + (uint32_t)n_stages * kStageBytes;
    L.total = L.off_misc + (uint32_t)((sizeof(Misc) + 127) / 128 * 128);
    return L;
}

__device__ __forceinline__ uint32_t row_offset(int c)
{
    return (c & 1) ? kOddRows + (uint32_t)(c >> 1) * 256u : (uint32_t)(c >> 1) * 256u;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v)
{
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Four int8 codes -> four f16 values (exact): bias the bytes to u = code+128,
// place them as the low mantissa bits of 1024 (0x6400), subtract 1152.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const uint32_t bias = 0x64806480u;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__device__ __forceinline__ int ordered_key(float f)
{
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}

__device__ __forceinline__ float from_ordered_key(int k)
{
    return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff);
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- work list

// Non-empty (sequence, KV head, chunk) items in sequence-major order; each
// CTA takes a contiguous range.  Producer and consumers walk it identically.
struct Cursor {
    int b, g, c, nch, start, n;
    int remaining;
};

__device__ inline int seq_chunks(const Params &p, int b, int *start, int *n)
{
    seq_range(p, b, start, n);
    return *n > 0 ? (*n + p.chunk_cells - 1) / p.chunk_cells : 0;
}

__device__ inline void cursor_init(const Params &p, Cursor &cur)
{
    long long total = 0;
    int s, n;
    for (int b = 0; b < p.n_seq; ++b) total += (long long)p.G * seq_chunks(p, b, &s, &n);
    const long long per = (total + gridDim.x - 1) / gridDim.x;
    long long lo = per * blockIdx.x;
    const long long hi = min(lo + per, total);
    cur.remaining = lo < hi ? (int)(hi - lo) : 0;
    cur.b = 0;
    cur.g = cur.c = 0;
    cur.nch = 0;
    if (cur.remaining == 0) return;
    for (int b = 0; b < p.n_seq; ++b) {
        const int nch = seq_chunks(p, b, &s, &n);
        const long long items = (long long)p.G * nch;
        if (lo < items) {
            cur.b = b;
            cur.nch = nch;
            cur.start = s;
            cur.n = n;
            cur.g = (int)(lo / nch);
            cur.c = (int)(lo % nch);
            return;
        }
        lo -= items;
    }
    cur.remaining = 0;
}

__device__ inline void cursor_next(const Params &p, Cursor &cur)
{
    if (--cur.remaining <= 0) return;
    if (++cur.c < cur.nch) return;
    cur.c = 0;
    if (++cur.g < p.G) return;
    cur.g = 0;
    int s, n;
    for (int b = cur.b + 1; b < p.n_seq; ++b) {
        const int nch = seq_chunks(p, b, &s, &n);
        if (nch > 0) {
            cur.b = b;
            cur.nch = nch;
            cur.start = s;
            cur.n = n;
            return;
        }
    }
    cur.remaining = 0;
}

// ---------------------------------------------------------------- producer

__device__ void run_producer(const Params &p, uint8_t *smem, const Layout &L, Misc &ms)
{
    const int lane = threadIdx.x & 31;
    const uint32_t raw_base = smem_u32(smem + L.off_raw);
    uint32_t op = 0;
    Cursor cur;
    cursor_init(p, cur);
    for (; cur.remaining > 0; cursor_next(p, cur)) {
        const int c0 = cur.c * p.chunk_cells;
        const int nc = min(p.chunk_cells, cur.n - c0);
        const size_t kv_base = ((size_t)cur.b * p.G + cur.g) * p.pool_cells;
        for (int gs = 0; gs < nc; gs += kGroupCells) {
            const int gn = min(kGroupCells, nc - gs);
            const int tiles = (gn + kTile - 1) / kTile;
            int slots[kMaxTiles][4];
#pragma unroll
            for (int t = 0; t < kMaxTiles; ++t) {
                int pos[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = t * kTile + lane * 4 + e;
                    pos[e] = (t < tiles && i < gn) ? __ldg(p.sel + cur.start + c0 + gs + i) : INT_MIN;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    slots[t][e] = pos[e] == INT_MIN ? -1 : resolve_slot(p, cur.b, pos[e]);
            }
            for (int kind = 0; kind < 2; ++kind) {
                for (int t = 0; t < tiles; ++t, ++op) {
                    const uint32_t s = op % L.n_stages;
                    const uint32_t round = op / L.n_stages;
                    if (ms.abort) continue; // stop issuing copies after a timeout
                    if (!mbar_wait(&ms.empty[s], (round & 1) ^ 1)) {
                        atomicExch(&ms.abort, 1);
                        raise_status(p, QSA_STATUS_TIMEOUT);
                        continue;
                    }
                    const uint32_t st = raw_base + s * kStageBytes;
                    int sl[4]; // this tile's slots (kept in registers: t is 0 or 1)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sl[e] = t == 0 ? slots[0][e] : slots[1][e];
                    int nvalid = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) nvalid += sl[e] >= 0;
                    if (kind == 0) {
                        const int c = lane * 4;
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(st + kStageSlots + c * 4),
                                     "r"(sl[0]), "r"(sl[1]), "r"(sl[2]), "r"(sl[3])
                                     : "memory");
                    }
                    __syncwarp();
                    const int total = __reduce_add_sync(0xffffffffu, nvalid);
                    if (lane == 0) mbar_arrive_expect_tx(&ms.full[s], (uint32_t)total * 256u);
                    const int8_t *pool = kind == 0 ? p.k_pool : p.v_pool;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = lane * 4 + e;
                        const int slot = sl[e];
                        if (slot < 0) continue;
                        bulk_g2s(smem + L.off_raw + s * kStageBytes + row_offset(c),
                                 pool + (kv_base + slot) * kHeadDim, 256, &ms.full[s]);
                        if (kind == 0) {
                            cp_async4(st + kStageKs + c * 4, p.k_scale + kv_base + slot);
                            cp_async4(st + kStageVs + c * 4, p.v_scale + kv_base + slot);
                        }
                    }
                    cp_async_arrive_noinc(&ms.full[s]);
                }
            }
        }
    }
    // After a timeout the consumers stop waiting; before the CTA may exit,
    // wait (bounded) for the copies this warp issued into the last stages.
    if (ms.abort) {
        const uint32_t n = op < L.n_stages ? op : L.n_stages;
        for (uint32_t i = 1; i <= n; ++i) {
            const uint32_t k = op - i;
            mbar_wait(&ms.full[k % L.n_stages], (k / L.n_stages) & 1, 1u << 22);
        }
    }
}

// ---------------------------------------------------------------- consumers

// Dequantise one raw stage (128 rows) into the f16 tile.  32 threads cover
// two rows x sixteen 16-byte pieces; even and odd rows sit in regions 64 B
// apart modulo 128, so both the reads and the swizzled writes are free of
// bank conflicts.
__device__ __forceinline__ void convert_tile(uint32_t stage, uint32_t tile, int cw, int lane)
{
    const int qlo = lane & 3, rsel = (lane >> 2) & 1, qhi = lane >> 3;
    const int q = qhi * 4 + qlo;
#pragma unroll 4
    for (int it = 0; it < 8; ++it) {
        const int rp = cw * 8 + it;
        const int row = 2 * rp + rsel;
        const uint4 raw = lds128(stage + (rsel ? kOddRows : 0u) + (uint32_t)rp * 256u + q * 16u);
        uint4 a, b;
        i8x4_to_f16x4(raw.x, a.x, a.y);
        i8x4_to_f16x4(raw.y, a.z, a.w);
        i8x4_to_f16x4(raw.z, b.x, b.y);
        i8x4_to_f16x4(raw.w, b.z, b.w);
        sts128(tile + kmajor_sw128_off(row, 16 * q, kTile), a);
        sts128(tile + kmajor_sw128_off(row, 16 * q + 8, kTile), b);
    }
}

__device__ __forceinline__ void load_queries(const Params &p, uint32_t sq, int b, int g, int N, int ct)
{
    const int GH = p.G * p.H;
    for (int e = ct; e < N * 32; e += kConsumers) {
        const int r = e >> 5, piece = e & 31;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < p.R) {
            const int t = r / p.H, j = r % p.H;
            const size_t off = (((size_t)b * p.T + t) * GH + (size_t)g * p.H + j) * kHeadDim + piece * 8;
            float f[8];
            if (p.q_bf16) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) + off);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    f[2 * e2] = bf16_bits_to_f32(w[e2] & 0xffff);
                    f[2 * e2 + 1] = bf16_bits_to_f32(w[e2] >> 16);
                }
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(p.q) + off);
                const float4 x = src[0], y = src[1];
                f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
                f[4] = y.x; f[5] = y.y; f[6] = y.z; f[7] = y.w;
            }
            __half2 h0 = __floats2half2_rn(f[0], f[1]), h1 = __floats2half2_rn(f[2], f[3]);
            __half2 h2 = __floats2half2_rn(f[4], f[5]), h3 = __floats2half2_rn(f[6], f[7]);
            v.x = *reinterpret_cast<uint32_t *>(&h0);
            v.y = *reinterpret_cast<uint32_t *>(&h1);
            v.z = *reinterpret_cast<uint32_t *>(&h2);
            v.w = *reinterpret_cast<uint32_t *>(&h3);
        }
        sts128(sq + kmajor_sw128_off(r, piece * 8, N), v);
    }
}

template <int N>
__device__ void run_consumers(const Params &p, uint8_t *smem, const Layout &L, Misc &ms)
{
    constexpr int NH = N / 2;                   // columns per warp half
    constexpr int NHP = NH <= 8 ? 8 : (NH <= 16 ? 16 : 32);
    const int ct = threadIdx.x - 32;            // consumer thread 0..255
    const int cw = ct >> 5, lane = ct & 31;
    const int qd = (cw + 1) & 3;                // TMEM lane quadrant of this warp
    const int ch = cw >> 2;                     // column half / d half
    const uint32_t s_kv = smem_u32(smem + L.off_kv);
    const uint32_t s_q = smem_u32(smem + L.off_q);
    const uint32_t s_p = smem_u32(smem + L.off_p);
    const uint32_t raw_base = smem_u32(smem + L.off_raw);
    const uint32_t tmem = ms.tmem;
    const uint32_t t_lane = (uint32_t)(32 * qd) << 16;
    const uint32_t o_base = kMaxTiles * N;
    const uint32_t idesc_s = idesc_f16(128, N, false, false, false, false);
    const uint32_t idesc_o = idesc_f16(128, N, false, false, true, false);

    uint32_t op = 0, mma_phase = 0;
    int cur_bg = -1;

    auto wait_mma = [&]() {
        if (!ms.abort && !mbar_wait(&ms.mma, mma_phase)) {
            atomicExch(&ms.abort, 1);
            raise_status(p, QSA_STATUS_TIMEOUT);
        }
        mma_phase ^= 1;
        tc_fence_after();
    };
    auto wait_full = [&](uint32_t s, uint32_t round) {
        if (!ms.abort && !mbar_wait(&ms.full[s], round & 1)) {
            atomicExch(&ms.abort, 1);
            raise_status(p, QSA_STATUS_TIMEOUT);
        }
    };

    Cursor cur;
    cursor_init(p, cur);
    for (; cur.remaining > 0; cursor_next(p, cur)) {
        const int c0 = cur.c * p.chunk_cells;
        const int nc = min(p.chunk_cells, cur.n - c0);
        const int bg = cur.b * p.G + cur.g;
        if (bg != cur_bg) {
            load_queries(p, s_q, cur.b, cur.g, N, ct);
            fence_proxy_async_smem();
            cur_bg = bg;
        }
        if (ct < 64) {
            ms.row_mrun[ct] = -INFINITY;
            ms.row_lrun[ct] = 0.f;
        }
        for (int gs = 0; gs < nc; gs += kGroupCells) {
            const int gn = min(kGroupCells, nc - gs);
            const int tiles = (gn + kTile - 1) / kTile;
            // ---- scores: one K tile at a time
            for (int t = 0; t < tiles; ++t, ++op) {
                const uint32_t s = op % L.n_stages, round = op / L.n_stages;
                const uint32_t st = raw_base + s * kStageBytes;
                wait_full(s, round);
                convert_tile(st, s_kv, cw, lane);
                if (ct < kTile) {
                    const int slot = *reinterpret_cast<const int *>(smem + L.off_raw + s * kStageBytes + kStageSlots + ct * 4);
                    ms.cell_slot[t][ct] = slot;
                    ms.cell_ks[t][ct] = *reinterpret_cast<const float *>(smem + L.off_raw + s * kStageBytes + kStageKs + ct * 4) * p.scale_log2;
                    ms.cell_vs[t][ct] = *reinterpret_cast<const float *>(smem + L.off_raw + s * kStageBytes + kStageVs + ct * 4);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                consumer_sync();
                tc_fence_after();
                if (ct == 0) {
                    mbar_arrive(&ms.empty[s]);
#pragma unroll
                    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                        const uint64_t ad = smem_desc(s_kv + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = smem_desc(s_q + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
                        mma_f16_ss(tmem + t * N, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&ms.mma);
                }
                wait_mma();
            }
            // ---- softmax over the group
            const int cell = 32 * qd + lane;
            float mx[NH];
#pragma unroll
            for (int j = 0; j < NH; ++j) mx[j] = -INFINITY;
            float vsabs = 0.f;
            for (int t = 0; t < tiles; ++t) {
                float sv[NH];
#pragma unroll
                for (int j = 0; j < NH; j += 8) tmem_ld8(tmem + t_lane + t * N + ch * NH + j, sv + j);
                tmem_wait_ld();
                const bool ok = ms.cell_slot[t][cell] >= 0;
                const float ksc = ms.cell_ks[t][cell];
                if (ok) vsabs = fmaxf(vsabs, fabsf(ms.cell_vs[t][cell]));
#pragma unroll
                for (int j = 0; j < NH; ++j) mx[j] = fmaxf(mx[j], ok ? sv[j] * ksc : -INFINITY);
            }
#pragma unroll
            for (int j = 0; j < NH; ++j) {
                const int key = __reduce_max_sync(0xffffffffu, ordered_key(mx[j]));
                if (lane == j) ms.red_max[ch][qd][j] = from_ordered_key(key);
            }
            {
                const unsigned u = __reduce_max_sync(0xffffffffu, __float_as_uint(vsabs));
                if (lane == 0) ms.red_vs[ch][qd] = __uint_as_float(u);
            }
            tc_fence_before();
            consumer_sync();
            tc_fence_after();
            float m2[NH];
#pragma unroll
            for (int j = 0; j < NH; ++j)
                m2[j] = fmaxf(fmaxf(ms.red_max[ch][0][j], ms.red_max[ch][1][j]),
                              fmaxf(ms.red_max[ch][2][j], ms.red_max[ch][3][j]));
            float sigma = fmaxf(fmaxf(ms.red_vs[ch][0], ms.red_vs[ch][1]), fmaxf(ms.red_vs[ch][2], ms.red_vs[ch][3]));
            if (!(sigma > 0.f)) sigma = 1.f;
            const float inv_sigma = 1.f / sigma;
            float ls[NHP];
#pragma unroll
            for (int j = 0; j < NHP; ++j) ls[j] = 0.f;
            for (int t = 0; t < tiles; ++t) {
                float sv[NH];
#pragma unroll
                for (int j = 0; j < NH; j += 8) tmem_ld8(tmem + t_lane + t * N + ch * NH + j, sv + j);
                tmem_wait_ld();
                const bool ok = ms.cell_slot[t][cell] >= 0;
                const float ksc = ms.cell_ks[t][cell];
                const float vsn = ok ? ms.cell_vs[t][cell] * inv_sigma : 0.f;
                const uint32_t ptile = s_p + t * (N * kTile * 2);
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    const float pr = ok ? fast_exp2(sv[j] * ksc - m2[j]) : 0.f;
                    ls[j] += pr;
                    const __half h = __float2half_rn(pr * vsn);
                    sts16(ptile + kmajor_sw128_off(ch * NH + j, cell, N), *reinterpret_cast<const uint16_t *>(&h));
                }
            }
            // reduce-scatter of the NH column sums over the warp's 32 cells
#pragma unroll
            for (int o = 16, cnt = NHP; o >= 1; o >>= 1) {
                if (cnt > 1) {
                    const int half = cnt / 2;
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        const float send = up ? ls[i] : ls[i + half];
                        const float keep = up ? ls[i + half] : ls[i];
                        ls[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                    cnt = half;
                } else {
                    ls[0] += __shfl_xor_sync(0xffffffffu, ls[0], o);
                }
            }
            {
                constexpr int lanes_per_col = 32 / NHP;
                const int col = lane / lanes_per_col;
                if (lane % lanes_per_col == 0 && col < NH) ms.red_sum[ch][qd][col] = ls[0];
            }
            if (ct == 0) ms.sigma = sigma;
            fence_proxy_async_smem();
            tc_fence_before();
            consumer_sync();
            tc_fence_after();
            // per-row group values and their combination with earlier groups
            if (ct < N) {
                const int r = ct, hr = r / NH, jr = r % NH;
                const float mg = fmaxf(fmaxf(ms.red_max[hr][0][jr], ms.red_max[hr][1][jr]),
                                       fmaxf(ms.red_max[hr][2][jr], ms.red_max[hr][3][jr]));
                const float lg = ((ms.red_sum[hr][0][jr] + ms.red_sum[hr][1][jr]) + ms.red_sum[hr][2][jr]) +
                                 ms.red_sum[hr][3][jr];
                const float mr = ms.row_mrun[r];
                const float mn = fmaxf(mr, mg);
                float fa = 0.f, fb = 0.f;
                if (mn > -INFINITY) {
                    fa = mr == mn ? 1.f : (mr > -INFINITY ? fast_exp2(mr - mn) : 0.f);
                    fb = mg == mn ? 1.f : (mg > -INFINITY ? fast_exp2(mg - mn) : 0.f);
                }
                ms.row_fa[r] = fa;
                ms.row_fb[r] = fb;
                ms.row_mrun[r] = mn;
                ms.row_lrun[r] = ms.row_lrun[r] * fa + lg * fb;
            }
            // ---- P.V: one V tile at a time
            for (int t = 0; t < tiles; ++t, ++op) {
                const uint32_t s = op % L.n_stages, round = op / L.n_stages;
                const uint32_t st = raw_base + s * kStageBytes;
                wait_full(s, round);
                convert_tile(st, s_kv, cw, lane);
                fence_proxy_async_smem();
                tc_fence_before();
                consumer_sync();
                tc_fence_after();
                if (ct == 0) {
                    mbar_arrive(&ms.empty[s]);
                    const uint32_t ptile = s_p + t * (N * kTile * 2);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk) {
                            const uint64_t ad = smem_desc(s_kv + (2 * h) * (kTile * 128) + kk * 2048, kTile * 128, 1024);
                            const uint64_t bd = smem_desc(ptile + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
                            mma_f16_ss(tmem + o_base + h * N, ad, bd, idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(&ms.mma);
                }
                wait_mma();
            }
            // ---- fold the group's O into the chunk partial.  The first group
            // writes it; a later group (chunks longer than 256 cells) rescales
            // the partial already written by this thread and adds to it.
            {
                const int d = ch * 128 + 32 * qd + lane;
                const size_t base = (((size_t)cur.b * p.G + cur.g) * p.n_chunks + cur.c) * p.R;
                const float sg = ms.sigma;
#pragma unroll
                for (int j0 = 0; j0 < N; j0 += 16) {
                    float ov[16];
                    tmem_ld16(tmem + t_lane + o_base + ch * N + j0, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int r = j0 + i;
                        if (r >= p.R) continue;
                        float* dst = p.part_o + (base + r) * kHeadDim + d;
                        float v = ov[i] * sg * ms.row_fb[r];
                        if (gs > 0) v = fmaf(*dst, ms.row_fa[r], v);
                        *dst = v;
                    }
                }
            }
            tc_fence_before();
            consumer_sync();
            tc_fence_after();
        }
        // ---- item epilogue: the chunk's max and denominator
        if (ct < p.R) {
            const size_t base = (((size_t)cur.b * p.G + cur.g) * p.n_chunks + cur.c) * p.R;
            p.part_m[base + ct] = ms.row_mrun[ct] * kLn2;
            p.part_l[base + ct] = ms.row_lrun[ct];
        }
        consumer_sync();
    }
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1) qsa_chunk_tc_kernel(const Params p, int n_stages)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = ((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw);
    uint8_t *smem = smem_raw + pad;
    const Layout L = make_layout(N, n_stages);
    Misc &ms = *reinterpret_cast<Misc *>(smem + L.off_misc);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < n_stages; ++s) {
            mbar_init(&ms.full[s], 33);
            mbar_init(&ms.empty[s], 1);
        }
        mbar_init(&ms.mma, 1);
        ms.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&ms.tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0)
        run_producer(p, smem, L, ms);
    else
        run_consumers<N>(p, smem, L, ms);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(ms.tmem, kTmemCols);
}

template <int N>
cudaError_t launch_n(const Params &p, cudaStream_t stream)
{
    int dev = 0, sms = 0, max_smem = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    int n_stages = 3;
    uint32_t bytes = make_layout(N, n_stages).total + 1024;
    if ((int)bytes > max_smem) {
        n_stages = 2;
        bytes = make_layout(N, n_stages).total + 1024;
    }
    if ((int)bytes > max_smem) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(qsa_chunk_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)bytes)) != cudaSuccess)
        return e;
    const long long items = (long long)p.n_seq * p.G * p.n_chunks;
    const int grid = (int)(items < (long long)sms ? items : (long long)sms);
    qsa_chunk_tc_kernel<N><<<grid, kThreads, bytes, stream>>>(p, n_stages);
    return cudaGetLastError();
}

} // namespace

bool chunk_tc_supports(const Params &p) { return p.R <= 64; }

cudaError_t launch_chunk_tc(const Params &p, cudaStream_t stream)
{
    if (p.n_chunks == 0) return cudaSuccess;
    const int N = (p.R + 15) / 16 * 16;
    switch (N) {
    case 16: return launch_n<16>(p, stream);
    case 32: return launch_n<32>(p, stream);
    case 48: return launch_n<48>(p, stream);
    case 64: return launch_n<64>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace qsa
