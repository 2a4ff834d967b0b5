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
// Two persistent CTAs of 8 warps share each SM (about 110 KB of shared
// memory and 256 TMEM columns each), so one CTA's dependent phases overlap
// the other's.  A CTA walks a contiguous range of non-empty (sequence, KV
// head, chunk) items as a sequence of ops: for every group of up to 256
// cells (two M tiles sharing one max), its K tiles, then its V tiles.
//   gather   each op's 128 rows (256 B each) are loaded straight into
//            registers with 16-byte read-only loads one op ahead (8 x 16 B
//            per thread, issued as soon as the previous op is converted);
//            16 lanes cover a row, so every load instruction moves two whole
//            rows; the op after that is prefetched into L2 at the same time,
//            so the register loads mostly hit L2;
//   resolve  list entry -> page slot (a1) runs two groups ahead: list reads
//            at a group's first K op, page-table reads after its max pass,
//            the checked slots stored in a small ring at the group's end;
//   convert  registers -> f16 tile in the tensor cores' 128-byte-swizzled
//            layout (the lane mapping makes the stores conflict-free);
//   MMA      one thread issues tcgen05.mma; completion on an mbarrier;
//   softmax  warp (quadrant q, half h) owns cells 32q..32q+31 and half the
//            rows, eight rows at a time: max via redux, P built per tile
//            right before its P.V MMA, sums via a reduce-scatter butterfly,
//            all in a fixed order, so partials are bit-identical run to run.
//
// The only wait that is not a CTA barrier is the MMA-completion wait; it is
// bounded, and a wait that runs out raises QSA_STATUS_TIMEOUT and the kernel
// runs to its end without further waiting.
#include <cuda_fp16.h>

#include "qsa_internal.cuh"
#include "qsa_sm100.cuh"

namespace qsa {
namespace {

using namespace sm100;

constexpr int kTile = 128;          // cells per MMA tile (M)
constexpr int kMaxTiles = 2;        // tiles per softmax group
constexpr int kGroupCells = kTile * kMaxTiles;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlotRing = 4;        // groups of resolved slots kept
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTileF16Bytes = kTile * kHeadDim * 2; // 64 KB

struct Layout {
    uint32_t off_kv, off_q, off_p, off_misc, total;
};

// Position in the work list (see cursor_init_warp / cursor_next).
struct Cursor {
    int b, g, c, nch, start, n;
    int remaining;
};

// Misc area: slot ring, per-group cell info, reduction scratch, per-row values.
struct Misc {
    int32_t ring[kSlotRing][kGroupCells];
    int32_t cell_slot[kMaxTiles][kTile];
    float cell_ks[kMaxTiles][kTile];
    float cell_vs[kMaxTiles][kTile];
    float red_max[2][32][4]; // [row half][row within half][lane quadrant]
    float red_sum[2][32][4];
    float red_vs[kWarps];
    float row_fa[64], row_fb[64], row_mrun[64], row_lrun[64];
    int32_t abort;
    uint32_t tmem;
    Cursor first; // this CTA's first item
    uint64_t mma;
};

__host__ __device__ inline Layout make_layout(int N)
{
    Layout L;
    L.off_kv = 0;
    L.off_q = kTileF16Bytes;
    L.off_p = L.off_q + (uint32_t)N * kHeadDim * 2;
    L.off_misc = L.off_p + (uint32_t)N * kTile * 2;
    L.total = L.off_misc + (uint32_t)((sizeof(Misc) + 127) / 128 * 128);
    return L;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
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

// NC consecutive columns of tensor memory (a multiple of 4) into v.
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float *v)
{
#pragma unroll
    for (int j = 0; j + 8 <= NC; j += 8) tmem_ld8(taddr + j, v + j);
    if (NC % 8) tmem_ld4(taddr + (NC / 8) * 8, v + (NC / 8) * 8);
}

// ---------------------------------------------------------------- work list

// Non-empty (sequence, KV head, chunk) items in sequence-major order; each
// CTA takes a contiguous range (consecutive chunks share their queries).

__device__ inline int seq_chunks(const Params &p, int b, int *start, int *n)
{
    seq_range(p, b, start, n);
    return *n > 0 ? (*n + p.chunk_cells - 1) / p.chunk_cells : 0;
}

// Position of this CTA's first item, computed by one full warp: lanes read
// the sequences' list offsets in parallel, a warp scan finds the sequence
// that holds item `lo`.
__device__ inline void cursor_init_warp(const Params &p, Cursor &cur, int lane)
{
    long long total = 0;
    int s, n;
    for (int b = lane; b < p.n_seq; b += 32) total += (long long)p.G * seq_chunks(p, b, &s, &n);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    const long long per = (total + gridDim.x - 1) / gridDim.x;
    const long long lo = per * blockIdx.x;
    const long long hi = min(lo + per, total);
    cur.remaining = lo < hi ? (int)(hi - lo) : 0;
    cur.b = cur.g = cur.c = cur.nch = cur.start = cur.n = 0;
    if (cur.remaining == 0) return;
    long long before = 0; // items of the sequences already passed
    for (int b0 = 0; b0 < p.n_seq; b0 += 32) {
        const int b = b0 + lane;
        int st = 0, len = 0, nch = 0;
        if (b < p.n_seq) nch = seq_chunks(p, b, &st, &len);
        const long long items = (long long)p.G * nch;
        long long incl = items;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const long long excl = incl - items;
        const unsigned hit = __ballot_sync(0xffffffffu, items > 0 && before + excl <= lo && lo < before + incl);
        if (hit) {
            const int src = __ffs(hit) - 1;
            const long long off = lo - before - __shfl_sync(0xffffffffu, excl, src);
            cur.b = b0 + src;
            cur.nch = __shfl_sync(0xffffffffu, nch, src);
            cur.start = __shfl_sync(0xffffffffu, st, src);
            cur.n = __shfl_sync(0xffffffffu, len, src);
            cur.g = (int)(off / cur.nch);
            cur.c = (int)(off % cur.nch);
            return;
        }
        before += __shfl_sync(0xffffffffu, incl, 31);
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

// The ops of the work range: for every group (up to two tiles of one
// chunk), its K tiles, then its V tiles.  Groups are numbered by gi in the
// same order everywhere (slot ring index = gi % kSlotRing).
struct OpIter {
    Cursor cur;
    int nc;      // cells of the current item (chunk)
    int gs;      // first cell of the current group within the item
    int tiles;   // tiles of the current group
    int kind;    // 0 = K tile, 1 = V tile
    int t;       // tile within the group
    uint32_t gi; // group counter
    bool valid;
};

__device__ inline void op_setup_item(const Params &p, OpIter &it)
{
    it.nc = min(p.chunk_cells, it.cur.n - it.cur.c * p.chunk_cells);
    it.gs = 0;
    it.kind = 0;
    it.t = 0;
    it.tiles = (min(kGroupCells, it.nc) + kTile - 1) / kTile;
}

__device__ inline void op_init(const Params &p, OpIter &it, const Cursor &first)
{
    it.cur = first;
    it.gi = 0;
    it.valid = it.cur.remaining > 0;
    if (it.valid) op_setup_item(p, it);
}

// Advance to the first op of the next group.
__device__ inline void op_next_group(const Params &p, OpIter &it)
{
    it.t = 0;
    it.kind = 0;
    ++it.gi;
    it.gs += kGroupCells;
    if (it.gs < it.nc) {
        it.tiles = (min(kGroupCells, it.nc - it.gs) + kTile - 1) / kTile;
        return;
    }
    cursor_next(p, it.cur);
    it.valid = it.cur.remaining > 0;
    if (it.valid) op_setup_item(p, it);
}

__device__ inline void op_next(const Params &p, OpIter &it)
{
    if (++it.t < it.tiles) return;
    it.t = 0;
    if (++it.kind < 2) return;
    op_next_group(p, it);
}

// ---------------------------------------------------------------- phases

// Step a1 for one cell of a group, split in three so the two dependent reads
// overlap other work: list entry, page entry, then the checks.
__device__ __forceinline__ int resolve_list(const Params &p, const OpIter &g, int i)
{
    if (!g.valid || i >= min(kGroupCells, g.nc - g.gs)) return INT_MIN;
    return __ldg(p.sel + g.cur.start + g.cur.c * p.chunk_cells + g.gs + i);
}

// INT_MIN marks a position outside the page table; -1 a cell past the group.
__device__ __forceinline__ int resolve_page(const Params &p, const OpIter &g, int pos)
{
    if (pos == INT_MIN) return -1;
    if (pos < 0 || pos >= p.page_table_len) return INT_MIN;
    return __ldg(p.page_table + (size_t)g.cur.b * p.page_table_len + pos);
}

__device__ __forceinline__ int resolve_check(const Params &p, int raw)
{
    if (raw == INT_MIN) {
        raise_status(p, QSA_STATUS_BAD_POSITION);
        return -1;
    }
    if (raw == -1) return -1;
    if (raw < 0 || raw >= p.pool_cells) {
        raise_status(p, QSA_STATUS_BAD_SLOT);
        return -1;
    }
    return raw;
}

// One op's rows in registers: warp w loads row pairs 8w..8w+7; lane
// (qhi, rsel, qlo) takes piece q = 4*qhi + qlo (16 B) of row 2*rp + rsel.
// Cells that are masked load nothing (zeros).  For a K op the first 128
// threads also load their cell's two scales.
struct OpRegs {
    uint4 raw[8];
    float ks, vs;
};

__device__ __forceinline__ void load_op(const Params &p, const Misc &ms, const OpIter &it, int tid,
                                        OpRegs &r)
{
    const int w = tid >> 5, lane = tid & 31;
    const int rsel = (lane >> 2) & 1, q = (lane >> 3) * 4 + (lane & 3);
    const int *tslots = ms.ring[it.gi % kSlotRing] + it.t * kTile;
    const size_t kv_base = ((size_t)it.cur.b * p.G + it.cur.g) * p.pool_cells;
    const int8_t *pool = (it.kind == 0 ? p.k_pool : p.v_pool) + kv_base * kHeadDim + q * 16;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int slot = tslots[2 * (8 * w + i) + rsel];
        r.raw[i] = slot >= 0 ? ldg_nc_v4(pool + (size_t)slot * kHeadDim) : make_uint4(0, 0, 0, 0);
    }
    r.ks = r.vs = 0.f;
    if (it.kind == 0 && tid < kTile) {
        const int slot = tslots[tid];
        if (slot >= 0) {
            r.ks = __ldg(p.k_scale + kv_base + slot);
            r.vs = __ldg(p.v_scale + kv_base + slot);
        }
    }
}

// Warm L2 with the rows (and, for a K op, the scales) of an op that is
// loaded into registers one op later: thread i prefetches 128-byte line
// i % 2 of row i / 2.  No registers or shared memory are held.
__device__ __forceinline__ void prefetch_op(const Params &p, const Misc &ms, const OpIter &it, int tid)
{
    const int *tslots = ms.ring[it.gi % kSlotRing] + it.t * kTile;
    const size_t kv_base = ((size_t)it.cur.b * p.G + it.cur.g) * p.pool_cells;
    const int slot = tslots[tid >> 1];
    if (slot >= 0) {
        const int8_t *row = (it.kind == 0 ? p.k_pool : p.v_pool) + (kv_base + slot) * kHeadDim + (tid & 1) * 128;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
        if (it.kind == 0) {
            const float *sc = (tid & 1) ? p.v_scale : p.k_scale;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(sc + kv_base + slot));
        }
    }
}

// Registers -> f16 tile: row = 2*(8w + i) + rsel, so row/8 = 2w + i/4 and
// row%8 = 2*(i%4) + rsel; the two 16-byte f16 chunks of piece q land in
// chunks 2*qlo and 2*qlo+1 of their 64-column block, XOR-swizzled by row%8.
__device__ __forceinline__ void convert_op(const OpRegs &r, uint32_t tile, int tid)
{
    const int w = tid >> 5, lane = tid & 31;
    const int qlo = lane & 3, rsel = (lane >> 2) & 1, qhi = lane >> 3;
    const uint32_t dst0 = tile + (uint32_t)qhi * (kTile * 128) + (uint32_t)(2 * w) * 1024u + (uint32_t)rsel * 128u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t r8 = 2u * (i & 3) + rsel;
        const uint32_t dst = dst0 + (uint32_t)(i >> 2) * 1024u + 2u * (i & 3) * 128u;
        uint4 a, b;
        i8x4_to_f16x4(r.raw[i].x, a.x, a.y);
        i8x4_to_f16x4(r.raw[i].y, a.z, a.w);
        i8x4_to_f16x4(r.raw[i].z, b.x, b.y);
        i8x4_to_f16x4(r.raw[i].w, b.z, b.w);
        sts128(dst + (((2u * qlo) ^ r8) << 4), a);
        sts128(dst + (((2u * qlo + 1u) ^ r8) << 4), b);
    }
}

__device__ __forceinline__ void cta_sync()
{
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Queries of (sequence b, KV head g) as the f16 B operand (rows >= R zero).
__device__ __forceinline__ void load_queries(const Params &p, uint32_t sq, int b, int g, int N, int tid)
{
    const int GH = p.G * p.H;
    for (int e = tid; e < N * 32; e += kThreads) {
        const int r = e >> 5, piece = e & 31;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < p.R) {
            const int t = r / p.H, j = r % p.H;
            const size_t off = (((size_t)b * p.T + t) * GH + (size_t)g * p.H + j) * kHeadDim + piece * 8;
            float f[8];
            if (p.q_bf16) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) + off);
                const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    f[2 * e2] = bf16_bits_to_f32(wv[e2] & 0xffff);
                    f[2 * e2 + 1] = bf16_bits_to_f32(wv[e2] >> 16);
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

// ---------------------------------------------------------------- kernel

template <int N>
__global__ void __launch_bounds__(kThreads, 2) qsa_chunk_tc_kernel(const Params p)
{
    constexpr int NH = N / 2; // rows per warp half (a multiple of 8)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = ((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw);
    uint8_t *smem = smem_raw + pad;
    const Layout L = make_layout(N);
    Misc &ms = *reinterpret_cast<Misc *>(smem + L.off_misc);
    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    const int qd = w & 3;  // TMEM lane quadrant of this warp
    const int ch = w >> 2; // row half (softmax) and d half (fold)
    const uint32_t s_kv = smem_u32(smem + L.off_kv);
    const uint32_t s_q = smem_u32(smem + L.off_q);
    const uint32_t s_p = smem_u32(smem + L.off_p);
    const uint32_t t_lane = (uint32_t)(32 * qd) << 16;
    const uint32_t o_base = kMaxTiles * N;
    const uint32_t idesc_s = idesc_f16(128, N, false, false, false, false);
    const uint32_t idesc_o = idesc_f16(128, N, false, false, true, false);
    const int cell = 32 * qd + lane; // softmax: this thread's cell within a tile

    if (tid == 0) {
        mbar_init(&ms.mma, 1);
        ms.abort = 0;
        fence_mbar_init();
    }
    if (w == 0) {
        tmem_alloc(&ms.tmem, kTmemCols);
        tmem_relinquish();
    }
    if (w == 1) cursor_init_warp(p, ms.first, lane);
    cta_sync();
    // the merge kernel may be scheduled now; it waits for this grid's results
    cudaTriggerProgrammaticLaunchCompletion();
    const uint32_t tmem = ms.tmem;
    const Cursor first = ms.first;
    uint32_t mma_phase = 0;
    auto wait_mma = [&]() {
        if (!ms.abort && !mbar_wait(&ms.mma, mma_phase)) {
            atomicExch(&ms.abort, 1);
            raise_status(p, QSA_STATUS_TIMEOUT);
        }
        mma_phase ^= 1;
        tc_fence_after();
    };

    // ---- resolve the first two groups (one per half of the threads)
    OpIter rg; // the group being resolved (two ahead of the one computed)
    op_init(p, rg, first);
    {
        OpIter g1 = rg;
        if (g1.valid) op_next_group(p, g1);
        const OpIter &mine = tid < kTile ? rg : g1;
        for (int i = tid & (kTile - 1); i < kGroupCells; i += kTile) {
            const int pos = resolve_list(p, mine, i);
            const int slot = resolve_check(p, resolve_page(p, mine, pos));
            if (mine.valid) ms.ring[mine.gi % kSlotRing][i] = slot;
        }
        rg = g1;
        if (rg.valid) op_next_group(p, rg);
    }
    __syncthreads();

    OpIter is, cs; // loads run one op ahead of the compute side
    op_init(p, is, first);
    op_init(p, cs, first);
    OpRegs rr; // the rows of the next op to convert
    if (is.valid) { load_op(p, ms, is, tid, rr); op_next(p, is); }
    if (is.valid) prefetch_op(p, ms, is, tid);

    int cur_bg = -1;
    int r_pos = INT_MIN, r_raw = -1; // this thread's cell of the group being resolved
    float sigma = 1.f, inv_sigma = 1.f;
    for (uint32_t op = 0; cs.valid; ++op) {
        const int t = cs.t;
        const bool last_tile = t == cs.tiles - 1;
        if (cs.kind == 0) {
            // ---- scores of one K tile
            if (t == 0) {
                if (tid < kGroupCells) r_pos = resolve_list(p, rg, tid);
                if (cs.gs == 0) {
                    const int bg = cs.cur.b * p.G + cs.cur.g;
                    if (bg != cur_bg) {
                        load_queries(p, s_q, cs.cur.b, cs.cur.g, N, tid);
                        cur_bg = bg;
                    }
                    if (tid < 64) {
                        ms.row_mrun[tid] = -INFINITY;
                        ms.row_lrun[tid] = 0.f;
                    }
                }
            }
            convert_op(rr, s_kv, tid);
            if (tid < kTile) {
                ms.cell_slot[t][tid] = ms.ring[cs.gi % kSlotRing][t * kTile + tid];
                ms.cell_ks[t][tid] = rr.ks * p.scale_log2;
                ms.cell_vs[t][tid] = rr.vs;
            }
            if (is.valid) {
                load_op(p, ms, is, tid, rr);
                op_next(p, is);
                if (is.valid) prefetch_op(p, ms, is, tid);
            }
            fence_proxy_async_smem();
            cta_sync();
            if (tid == 0) {
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint64_t ad = smem_desc(s_kv + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(s_q + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
                    mma_f16_ss(tmem + t * N, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&ms.mma);
            }
            wait_mma();
            if (last_tile) {
                // ---- max pass over the group, eight rows at a time: warp
                // (qd, ch) owns cells 32qd..32qd+31 and rows ch*NH..ch*NH+NH-1
                float vsabs = 0.f;
                for (int tt = 0; tt < cs.tiles; ++tt)
                    if (ms.cell_slot[tt][cell] >= 0) vsabs = fmaxf(vsabs, fabsf(ms.cell_vs[tt][cell]));
#pragma unroll
                for (int j0 = 0; j0 < NH; j0 += 8) {
                    float mx[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) mx[j] = -INFINITY;
                    for (int tt = 0; tt < cs.tiles; ++tt) {
                        float sv[8];
                        tmem_ld8(tmem + t_lane + tt * N + ch * NH + j0, sv);
                        tmem_wait_ld();
                        const bool ok = ms.cell_slot[tt][cell] >= 0;
                        const float ksc = ms.cell_ks[tt][cell];
#pragma unroll
                        for (int j = 0; j < 8; ++j) mx[j] = fmaxf(mx[j], ok ? __fmul_rn(sv[j], ksc) : -INFINITY);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int key = __reduce_max_sync(0xffffffffu, ordered_key(mx[j]));
                        if (lane == j) ms.red_max[ch][j0 + j][qd] = from_ordered_key(key);
                    }
                }
                {
                    const unsigned u = __reduce_max_sync(0xffffffffu, __float_as_uint(vsabs));
                    if (lane == 0) ms.red_vs[w] = __uint_as_float(u);
                }
                // the group two ahead: its page-table reads go out now
                if (tid < kGroupCells) r_raw = resolve_page(p, rg, r_pos);
                cta_sync();
                sigma = fmaxf(fmaxf(ms.red_vs[0], ms.red_vs[1]), fmaxf(ms.red_vs[2], ms.red_vs[3]));
                if (!(sigma > 0.f)) sigma = 1.f;
                inv_sigma = 1.f / sigma;
            }
        } else {
            // ---- P of one tile, then P.V
            {
                const bool ok = ms.cell_slot[t][cell] >= 0;
                const float ksc = ms.cell_ks[t][cell];
                const float vsn = ok ? ms.cell_vs[t][cell] * inv_sigma : 0.f;
#pragma unroll
                for (int j0 = 0; j0 < NH; j0 += 8) {
                    float sv[8], ls[8];
                    tmem_ld8(tmem + t_lane + t * N + ch * NH + j0, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 q4 = *reinterpret_cast<const float4 *>(ms.red_max[ch][j0 + j]);
                        const float m2 = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
                        // the same rounded product as in the max pass (no FMA
                        // contraction), so the max cell gets exactly 2^0 = 1
                        const float pr = ok ? fast_exp2(__fmul_rn(sv[j], ksc) - m2) : 0.f;
                        ls[j] = pr;
                        const __half h = __float2half_rn(pr * vsn);
                        sts16(s_p + kmajor_sw128_off(ch * NH + j0 + j, cell, N),
                              *reinterpret_cast<const uint16_t *>(&h));
                    }
                    // reduce-scatter of the eight row sums over the warp's 32 cells:
                    // lane pairs (4c, 4c+1, 4c+2, 4c+3) end with row j0 + c
#pragma unroll
                    for (int o = 16, cnt = 8; o >= 1; o >>= 1) {
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
                    if ((lane & 3) == 0) {
                        float &acc = ms.red_sum[ch][j0 + (lane >> 2)][qd];
                        acc = t == 0 ? ls[0] : acc + ls[0];
                    }
                }
            }
            convert_op(rr, s_kv, tid);
            if (is.valid) {
                load_op(p, ms, is, tid, rr);
                op_next(p, is);
                if (is.valid) prefetch_op(p, ms, is, tid);
            }
            fence_proxy_async_smem();
            cta_sync();
            if (tid == 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk) {
                        const uint64_t ad = smem_desc(s_kv + (2 * h) * (kTile * 128) + kk * 2048, kTile * 128, 1024);
                        const uint64_t bd = smem_desc(s_p + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
                        mma_f16_ss(tmem + o_base + h * N, ad, bd, idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&ms.mma);
            }
            wait_mma();
            if (last_tile) {
                // per-row group values and their combination with earlier groups
                if (tid < N) {
                    const int r = tid, hr = r / NH, jr = r % NH;
                    const float4 m4 = *reinterpret_cast<const float4 *>(ms.red_max[hr][jr]);
                    const float4 l4 = *reinterpret_cast<const float4 *>(ms.red_sum[hr][jr]);
                    const float mg = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
                    const float lg = ((l4.x + l4.y) + l4.z) + l4.w;
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
                // the group two ahead: checked slots into the ring
                if (tid < kGroupCells && rg.valid) ms.ring[rg.gi % kSlotRing][tid] = resolve_check(p, r_raw);
                if (rg.valid) op_next_group(p, rg);
                r_pos = INT_MIN;
                r_raw = -1;
                cta_sync();
                // ---- fold the group's O into the chunk partial.  The first
                // group writes it; a later group (chunks longer than 256
                // cells) rescales the partial this thread wrote and adds.
                {
                    const int d = ch * 128 + 32 * qd + lane;
                    const size_t base = (((size_t)cs.cur.b * p.G + cs.cur.g) * p.n_chunks + cs.cur.c) * p.R;
#pragma unroll
                    for (int j0 = 0; j0 < N; j0 += 16) {
                        float ov[16];
                        tmem_ld16(tmem + t_lane + o_base + ch * N + j0, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int r = j0 + i;
                            if (r >= p.R) continue;
                            float *dst = p.part_o + (base + r) * kHeadDim + d;
                            float v = ov[i] * sigma * ms.row_fb[r];
                            if (cs.gs > 0) v = fmaf(*dst, ms.row_fa[r], v);
                            *dst = v;
                        }
                    }
                }
                if (cs.gs + kGroupCells >= cs.nc && tid < p.R) {
                    // ---- item epilogue: the chunk's max and denominator
                    const size_t base = (((size_t)cs.cur.b * p.G + cs.cur.g) * p.n_chunks + cs.cur.c) * p.R;
                    p.part_m[base + tid] = ms.row_mrun[tid] * kLn2;
                    p.part_l[base + tid] = ms.row_lrun[tid];
                }
                cta_sync();
            }
        }
        op_next(p, cs);
    }
    cta_sync();
    if (w == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int N>
cudaError_t launch_n(const Params &p, cudaStream_t stream)
{
    int dev = 0, sms = 0, max_smem = 0, sm_smem = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
        return e;
    const uint32_t bytes = make_layout(N).total + 1024;
    if ((int)bytes > max_smem) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(qsa_chunk_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)bytes)) != cudaSuccess)
        return e;
    // two CTAs per SM when their shared memory fits (1 KB per CTA is reserved)
    const int per_sm = 2 * ((int)bytes + 1024) <= sm_smem ? 2 : 1;
    const long long items = (long long)p.n_seq * p.G * p.n_chunks;
    const long long slots = (long long)sms * per_sm;
    const int grid = (int)(items < slots ? items : slots);
    qsa_chunk_tc_kernel<N><<<grid, kThreads, bytes, stream>>>(p);
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
