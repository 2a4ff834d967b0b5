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
// One persistent CTA of 16 warps per SM walks a contiguous range of
// non-empty (sequence, KV head, chunk) items as a sequence of ops: for every
// group of up to 256 cells (two M tiles sharing one max), its K tiles, then
// its V tiles.  Every warp takes part in every phase:
//   gather   the rows of op k+2 are copied with 16-byte cp.async into a ring
//            of three raw stages while op k is computed (random 256-byte rows
//            need many warps issuing copies: one warp tops out near 8 GB/s
//            per SM; one TMA bulk copy per row was ~10x slower still);
//   resolve  list entry -> page slot (a1) runs two groups ahead: the list
//            reads are issued at a group's first K op, the page-table reads
//            after its softmax max pass, and the checked slots are stored at
//            the group's end;
//   convert  a raw stage becomes an f16 tile in the tensor cores'
//            128-byte-swizzled layout (no bank conflicts on either side);
//   MMA      one thread issues tcgen05.mma; completion on an mbarrier;
//   softmax  warp (quadrant q, quarter c) owns cells 32q..32q+31 of a tile
//            and a quarter of the rows: max via redux, sums via a
//            reduce-scatter butterfly, all in a fixed order, so partials are
//            bit-identical run to run.
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
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kSlotRing = 4;        // groups of resolved slots kept
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
    float red_max[4][4][16]; // [row quarter][lane quadrant][row within quarter]
    float red_sum[4][4][16];
    float red_vs[kWarps];
    float row_fa[64], row_fb[64], row_mrun[64], row_lrun[64];
    float sigma;
    int32_t abort;
    uint32_t tmem;
    Cursor first; // this CTA's first item
    uint64_t mma;
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

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

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

// Copies of one op into a raw stage: warp w moves rows 8w..8w+7, two per
// instruction (16 lanes x 16 B per 256-byte row).  For a K op the first 128
// threads also publish their cell's slot and copy its two scales.  Masked
// cells are not copied: their stale bytes are finite codes that get zero
// weight.
__device__ __forceinline__ void issue_op(const Params &p, uint8_t *smem, const Misc &ms,
                                         const OpIter &it, uint32_t st_off, int tid)
{
    const int w = tid >> 5, lane = tid & 31;
    const int *tslots = ms.ring[it.gi % kSlotRing] + it.t * kTile;
    const size_t kv_base = ((size_t)it.cur.b * p.G + it.cur.g) * p.pool_cells;
    const int8_t *pool = (it.kind == 0 ? p.k_pool : p.v_pool) + kv_base * kHeadDim + (lane & 15) * 16;
    const uint32_t st = smem_u32(smem) + st_off;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = 8 * w + 2 * i + (lane >> 4);
        const int slot = tslots[row];
        if (slot >= 0) cp_async16(st + row_offset(row) + (lane & 15) * 16, pool + (size_t)slot * kHeadDim);
    }
    if (it.kind == 0 && tid < kTile) {
        const int slot = tslots[tid];
        *reinterpret_cast<int *>(smem + st_off + kStageSlots + tid * 4) = slot;
        if (slot >= 0) {
            cp_async4(st + kStageKs + tid * 4, p.k_scale + kv_base + slot);
            cp_async4(st + kStageVs + tid * 4, p.v_scale + kv_base + slot);
        }
    }
}

// Dequantise one raw stage (128 rows) into the f16 tile.  Warp w converts
// row pairs 4w..4w+3; 32 threads cover two rows x sixteen 16-byte pieces.
// Even and odd rows sit in regions 64 B apart modulo 128, so both the reads
// and the swizzled writes are free of bank conflicts.
__device__ __forceinline__ void convert_tile(uint32_t stage, uint32_t tile, int w, int lane)
{
    const int qlo = lane & 3, rsel = (lane >> 2) & 1, qhi = lane >> 3;
    const int q = qhi * 4 + qlo;
    // row = 2*(4w + it) + rsel: row/8 = w and row%8 = 2*it + rsel
    const uint32_t src0 = stage + (rsel ? kOddRows : 0u) + (uint32_t)(w * 4) * 256u + q * 16u;
    const uint32_t dst0 = tile + (uint32_t)qhi * (kTile * 128) + (uint32_t)w * 1024u + (uint32_t)rsel * 128u;
    uint4 raw[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) raw[it] = lds128(src0 + it * 256u);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const uint32_t r8 = 2u * it + rsel;
        const uint32_t dst = dst0 + 2u * it * 128u;
        uint4 a, b;
        i8x4_to_f16x4(raw[it].x, a.x, a.y);
        i8x4_to_f16x4(raw[it].y, a.z, a.w);
        i8x4_to_f16x4(raw[it].z, b.x, b.y);
        i8x4_to_f16x4(raw[it].w, b.z, b.w);
        sts128(dst + (((2u * qlo) ^ r8) << 4), a);
        sts128(dst + (((2u * qlo + 1u) ^ r8) << 4), b);
    }
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

__device__ __forceinline__ void cta_sync()
{
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// ---------------------------------------------------------------- kernel

template <int N>
__global__ void __launch_bounds__(kThreads, 1) qsa_chunk_tc_kernel(const Params p, int n_stages)
{
    constexpr int NQ = N / 4;                   // rows per warp in the softmax
    constexpr int NQP = NQ <= 4 ? 4 : (NQ <= 8 ? 8 : 16);
    constexpr int NO = N / 2;                   // rows per thread in the fold
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = ((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw);
    uint8_t *smem = smem_raw + pad;
    const Layout L = make_layout(N, n_stages);
    Misc &ms = *reinterpret_cast<Misc *>(smem + L.off_misc);
    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    const int qd = w & 3;                       // TMEM lane quadrant of this warp
    const int rq = w >> 2;                      // softmax row quarter
    const int oh = (w >> 2) & 1, oc = w >> 3;   // fold: d half, row half
    const uint32_t s_kv = smem_u32(smem + L.off_kv);
    const uint32_t s_q = smem_u32(smem + L.off_q);
    const uint32_t s_p = smem_u32(smem + L.off_p);
    const uint32_t t_lane = (uint32_t)(32 * qd) << 16;
    const uint32_t o_base = kMaxTiles * N;
    const uint32_t idesc_s = idesc_f16(128, N, false, false, false, false);
    const uint32_t idesc_o = idesc_f16(128, N, false, false, true, false);
    const uint32_t ahead = (uint32_t)n_stages - 1; // ops whose copies are in flight

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

    // ---- resolve the first two groups; later groups are resolved two ahead
    OpIter rg; // the group being resolved
    op_init(p, rg, first);
    {
        OpIter g1 = rg; // threads 0..255 resolve group 0, threads 256..511 group 1
        if (g1.valid) op_next_group(p, g1);
        const OpIter &mine = tid < kGroupCells ? rg : g1;
        const int pos = resolve_list(p, mine, tid & (kGroupCells - 1));
        const int slot = resolve_check(p, resolve_page(p, mine, pos));
        if (mine.valid) ms.ring[mine.gi % kSlotRing][tid & (kGroupCells - 1)] = slot;
        rg = g1;
        if (rg.valid) op_next_group(p, rg);
    }
    __syncthreads();

    OpIter is, cs; // issue side (`ahead` ops in front) and compute side
    op_init(p, is, first);
    op_init(p, cs, first);
    for (uint32_t k = 0; k < ahead; ++k) {
        if (is.valid) {
            issue_op(p, smem, ms, is, L.off_raw + (k % n_stages) * kStageBytes, tid);
            op_next(p, is);
        }
        cp_async_commit();
    }

    int cur_bg = -1;
    int r_pos = INT_MIN, r_raw = -1; // this thread's cell of the group being resolved
    for (uint32_t op = 0; cs.valid; ++op) {
        if (is.valid) {
            issue_op(p, smem, ms, is, L.off_raw + ((op + ahead) % n_stages) * kStageBytes, tid);
            op_next(p, is);
        }
        cp_async_commit();
        if (ahead == 2)
            asm volatile("cp.async.wait_group 2;" ::: "memory");
        else
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        cta_sync(); // this op's rows and scales have landed, for every thread

        const uint32_t st_off = L.off_raw + (op % n_stages) * kStageBytes;
        const uint32_t st = smem_u32(smem) + st_off;
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
            convert_tile(st, s_kv, w, lane);
            if (tid < kTile) {
                const int slot = *reinterpret_cast<const int *>(smem + st_off + kStageSlots + tid * 4);
                ms.cell_slot[t][tid] = slot;
                ms.cell_ks[t][tid] = *reinterpret_cast<const float *>(smem + st_off + kStageKs + tid * 4) * p.scale_log2;
                ms.cell_vs[t][tid] = *reinterpret_cast<const float *>(smem + st_off + kStageVs + tid * 4);
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
                // ---- softmax over the group: warp (qd, rq) owns cells
                // 32qd..32qd+31 of each tile and rows rq*NQ..rq*NQ+NQ-1
                const int cell = 32 * qd + lane;
                float mx[NQ];
#pragma unroll
                for (int j = 0; j < NQ; ++j) mx[j] = -INFINITY;
                float vsabs = 0.f;
                for (int tt = 0; tt < cs.tiles; ++tt) {
                    float sv[NQ];
                    tmem_ld_cols<NQ>(tmem + t_lane + tt * N + rq * NQ, sv);
                    tmem_wait_ld();
                    const bool ok = ms.cell_slot[tt][cell] >= 0;
                    const float ksc = ms.cell_ks[tt][cell];
                    if (ok) vsabs = fmaxf(vsabs, fabsf(ms.cell_vs[tt][cell]));
#pragma unroll
                    for (int j = 0; j < NQ; ++j) mx[j] = fmaxf(mx[j], ok ? __fmul_rn(sv[j], ksc) : -INFINITY);
                }
#pragma unroll
                for (int j = 0; j < NQ; ++j) {
                    const int key = __reduce_max_sync(0xffffffffu, ordered_key(mx[j]));
                    if (lane == j) ms.red_max[rq][qd][j] = from_ordered_key(key);
                }
                {
                    const unsigned u = __reduce_max_sync(0xffffffffu, __float_as_uint(vsabs));
                    if (lane == 0) ms.red_vs[w] = __uint_as_float(u);
                }
                // the group two ahead: its page-table reads go out now
                if (tid < kGroupCells) r_raw = resolve_page(p, rg, r_pos);
                cta_sync();
                float m2[NQ];
#pragma unroll
                for (int j = 0; j < NQ; ++j)
                    m2[j] = fmaxf(fmaxf(ms.red_max[rq][0][j], ms.red_max[rq][1][j]),
                                  fmaxf(ms.red_max[rq][2][j], ms.red_max[rq][3][j]));
                float sigma = fmaxf(fmaxf(ms.red_vs[0], ms.red_vs[1]), fmaxf(ms.red_vs[2], ms.red_vs[3]));
                if (!(sigma > 0.f)) sigma = 1.f;
                const float inv_sigma = 1.f / sigma;
                float ls[NQP];
#pragma unroll
                for (int j = 0; j < NQP; ++j) ls[j] = 0.f;
                for (int tt = 0; tt < cs.tiles; ++tt) {
                    float sv[NQ];
                    tmem_ld_cols<NQ>(tmem + t_lane + tt * N + rq * NQ, sv);
                    tmem_wait_ld();
                    const bool ok = ms.cell_slot[tt][cell] >= 0;
                    const float ksc = ms.cell_ks[tt][cell];
                    const float vsn = ok ? ms.cell_vs[tt][cell] * inv_sigma : 0.f;
                    const uint32_t ptile = s_p + tt * (N * kTile * 2);
#pragma unroll
                    for (int j = 0; j < NQ; ++j) {
                        // the same rounded product as in the max pass (no FMA
                        // contraction), so the max cell gets exactly 2^0 = 1
                        const float pr = ok ? fast_exp2(__fmul_rn(sv[j], ksc) - m2[j]) : 0.f;
                        ls[j] += pr;
                        const __half h = __float2half_rn(pr * vsn);
                        sts16(ptile + kmajor_sw128_off(rq * NQ + j, cell, N),
                              *reinterpret_cast<const uint16_t *>(&h));
                    }
                }
                // reduce-scatter of the NQ row sums over the warp's 32 cells
#pragma unroll
                for (int o = 16, cnt = NQP; o >= 1; o >>= 1) {
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
                    constexpr int lanes_per_col = 32 / NQP;
                    const int col = lane / lanes_per_col;
                    if (lane % lanes_per_col == 0 && col < NQ) ms.red_sum[rq][qd][col] = ls[0];
                }
                if (tid == 0) ms.sigma = sigma;
                fence_proxy_async_smem();
                cta_sync();
                // per-row group values and their combination with earlier groups
                if (tid < N) {
                    const int r = tid, hr = r / NQ, jr = r % NQ;
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
            }
        } else {
            // ---- P.V of one V tile
            convert_tile(st, s_kv, w, lane);
            fence_proxy_async_smem();
            cta_sync();
            if (tid == 0) {
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
            if (last_tile) {
                // the group two ahead: checked slots into the ring
                if (tid < kGroupCells && rg.valid) ms.ring[rg.gi % kSlotRing][tid] = resolve_check(p, r_raw);
                if (rg.valid) op_next_group(p, rg);
                r_pos = INT_MIN;
                r_raw = -1;
                // ---- fold the group's O into the chunk partial.  The first
                // group writes it; a later group (chunks longer than 256
                // cells) rescales the partial this thread wrote and adds.
                {
                    const int d = oh * 128 + 32 * qd + lane;
                    const size_t base = (((size_t)cs.cur.b * p.G + cs.cur.g) * p.n_chunks + cs.cur.c) * p.R;
                    const float sg = ms.sigma;
                    float ov[NO];
                    tmem_ld_cols<NO>(tmem + t_lane + o_base + oh * N + oc * NO, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < NO; ++i) {
                        const int r = oc * NO + i;
                        if (r >= p.R) continue;
                        float *dst = p.part_o + (base + r) * kHeadDim + d;
                        float v = ov[i] * sg * ms.row_fb[r];
                        if (cs.gs > 0) v = fmaf(*dst, ms.row_fa[r], v);
                        *dst = v;
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
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    cta_sync();
    if (w == 0) tmem_dealloc(tmem, kTmemCols);
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
