// qsa_chunk_tc.cu -- tensor-core chunk kernel for decode windows (steps a1-a4).
//
// What it computes is the chunk step of "Strata PR #2220,
// attn_chunk_q8_v3_kernel": each chunk of the selected list yields partials
// (max m, sum of exponentials l, unnormalised P.V o) for every query row
// (T queries x H heads of one KV head).  Where a CTA takes several
// consecutive chunks of one (sequence, KV head) -- more chunks than CTAs --
// it accumulates up to eight of them into one partial: the same m, l, o
// over the run's cells, which the merge combines exactly as it would the
// chunks' own (the pages' split into chunks is the unit of work; partials
// per chunk only add stores and merge reads).  The pages' Turing kernel reads each
// cell once for all 12 heads and does the dot products with warp shuffles;
// here both contractions run on the 5th-generation tensor cores with the
// cells on the MMA's M dimension, because a decode window has only 12-80
// query rows:
//
//   S^T[cell][row] = K_code[cell][:] . Q[row][:]      M=128 cells, N=rows, K=256
//   O^T[d][row]   += V_code^T[d][cell] . P'^T[cell][row]   M=128 d (x2), N=rows, K=128 cells
//
// INT8 codes convert exactly to f16 (|code| <= 127).  The K scale (times the
// softmax scale and log2 e) multiplies the fp32 score after the MMA; the V
// scale, divided by a reference sigma, multiplies the probability before it
// is rounded to f16 (P' = p * v_scale / sigma), and sigma multiplies the fp32
// result.  A query element q is split into f16 parts hi = f16(q) and
// lo = f16(q - hi), and S = K.hi + K.lo (two MMAs per 16-wide contraction
// step into one fp32 accumulator): the query then carries about 22 bits
// instead of f16's 11.  Calls split their rows into blocks of at most 64
// (16-row multiples for one (sequence, KV head), 24 rows for several);
// windows of more than 64 rows with causal limits, which are not split, have
// no shared memory left for the low part and use hi alone.
//
// Probabilities are formed against a reference maximum per row (mref) that
// moves only when a score exceeds it by more than 2^8, so P' <= 2^8 * 16 stays
// far inside f16.  The reference lives from the first cell of a (sequence, KV
// head) pair that a CTA meets to its last one, across chunks.  Each tile the
// softmax threads vote, in one barrier-reduction, whether any score or V scale
// leaves the reference's range; only then (the first tile of a pair, or a
// score that jumps by 2^8) do they reduce the tile's true row maxima and move
// the reference, rescaling l and O.  Row sums and row maxima are kept per
// thread and reduced across the CTA once per run, where the partials are
// brought to the run's true maximum: m = max score, l = sum 2^(s - m),
// o = sum 2^(s - m) v_hat.
//
// One persistent CTA per SM walks a contiguous range of non-empty (sequence,
// KV head, chunk) items as a stream of 128-cell tiles, with warp roles that
// run concurrently and hand tiles over through mbarrier rings:
//
//   loader warps 0-7  (warp w: cells 32(w%4)+16(w/4)..+15).  A software
//            pipeline, one tile per step: list entries six tiles ahead,
//            page-table entries four ahead, slot checks, scale copies and L2
//            prefetch of the K/V rows two ahead (lanes 0-15 resolve one cell
//            each), 32-byte register loads of the rows one ahead; the current
//            tile's K codes go to tensor memory as the MMA's A operand
//            (tcgen05.st), its V codes to a double-buffered shared-memory
//            tile in the MN-major 128-byte-swizzled layout.
//   softmax warps 8-11 (warp q: tensor-memory lanes 32q..32q+31).  Per tile:
//            scores from tensor memory, the vote, P' as the second MMA's B
//            operand; at a chunk's end the partials.
//   S warp 12 (one thread) issues S = K.Q^T of each tile, and P.V warp 13
//            (one thread) O += V^T.P'^T, side by side; completion is
//            signalled by tcgen05.commit on the rings' barriers.
//
// Every wait is bounded; a wait that runs out raises QSA_STATUS_TIMEOUT and
// makes all later waits of the CTA return at once, so the kernel always
// ends.  Before the CTA leaves, each issuing thread waits (with a bound of its
// own) for its tensor-core operations and bulk copies, and each loader for its
// asynchronous copies, so nothing is in flight when tensor memory is freed.
#include <algorithm>
#include <cuda_fp16.h>
#include <float.h>

#include "qsa_internal.cuh"
#include "qsa_sm100.cuh"

namespace qsa {
namespace {

using namespace sm100;

constexpr int kTile = 128;                        // cells per tile (MMA M)
constexpr int kLoadWarps = 8;
constexpr int kSoftWarps = 4;
constexpr int kMmaWarp = kLoadWarps + kSoftWarps; // 12: issues S = K.Q^T
constexpr int kPvWarp = kMmaWarp + 1;             // 13: issues O += V^T.P'^T
constexpr int kThreads = (kPvWarp + 1) * 32;      // 448
constexpr int kLoadThreads = kLoadWarps * 32;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kResolveThreads = kLoadWarps * 16;  // loader lanes 0-15: one cell each
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxRows = kDecodeTcMaxRows;
constexpr uint32_t kStageBytes = kTile * kHeadDim * 2; // one f16 V tile, 64 KB
constexpr uint32_t kBarSoft = 1;                       // named barrier of the softmax warps
constexpr float kRescaleLog2 = 8.f; // the reference moves when a score exceeds it by 2^8
constexpr float kSigmaGrow = 16.f;  // ... sigma when a V scale exceeds 16 x sigma
constexpr long long kDrainCycles = 1ll << 30; // bound of the waits before the CTA leaves

// Position in the work list (see cursor_init_warp / cursor_next); lo and
// per (the CTA's first item and the items per CTA) are set for the first item.
struct Cursor {
    int b, g, c, nch, start, n;
    int remaining;
    int per;
    long long lo;
};

// Runs: a CTA accumulates up to kRunChunks consecutive chunks of one
// (sequence, KV head) in one partial (m, l, o), so the partials written and
// merged per row drop from the chunk count to about the number of CTAs that
// share the pair.  Item y (of a row block's list) starts a run when its
// offset in its CTA's range, y mod per, is a multiple of kRunChunks, or when
// it is its pair's first chunk.  The k-th run of a pair is stored at partial
// slot k; the pair's run count goes to part_runs for the merge.
constexpr int kRunChunks = 8;

struct Misc {
    // resolution rings (tile t in entry t % 4), filled by asynchronous copies
    int32_t rs_sel[4][kTile]; // list entries
    int32_t rs_pg[4][kTile];  // page-table entries (-1 masked, kBadPos out of range)
    int32_t rs_off[4][kTile]; // offset of the position in its page (pages of P > 1 cells)
    float rs_ks[4][kTile];    // k_scale, v_scale of the cell's slot (0 if masked)
    float rs_vs[4][kTile];
    uint8_t rs_ok[4][kTile];  // cell holds a valid slot
    uint8_t rs_r0[4][kTile];  // causal limits: the first query row that sees the cell (<= 80)
    uint8_t sc_r0[2][kTile];  // the same, handed to the softmax (two-entry ring)
    // softmax, after a vote: [warp][row] tile maxima, with the largest
    // |v_scale| at [kMaxRows]; the O factors of a moved reference.  (One
    // buffer: the next writer passes at least one barrier after the readers.)
    __align__(16) float red_max[4][kMaxRows + 4];
    __align__(16) float red_fac[kMaxRows + 4];
    // chunk ends: [warp][row] maxima and sums, the reference; and, per chunk
    // parity, the factor sigma * 2^(mref - m) the chunk's O is read out with
    __align__(16) float ch_max[4][kMaxRows];
    __align__(16) float ch_sum[4][kMaxRows];
    __align__(16) float ch_ref[kMaxRows];
    __align__(16) float st_fin[2][kMaxRows];
    __align__(16) float st_m[2][kMaxRows]; // the chunk's partial m and l, per chunk parity,
    __align__(16) float st_l[2][kMaxRows]; // stored with its O by the epilogue
    Cursor first;
    uint32_t tmem;
    int abort;
    uint64_t k_full[2], k_empty[2], s_done, pv_done;
    uint64_t q_full[2], q_empty[2];
    uint64_t v_full[2], v_empty[2], sc_full[2], sc_empty[2];
    uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2], o_full[2], o_empty[2];
};

template <int N>
struct Lay {
    static constexpr int PB = N <= 48 ? 2 : 1; // P' buffers
    static constexpr int QSF = N <= 64 ? 2 : 1; // query tile parts (hi, lo)
    // Query tile buffers: two (the next segment's tile loads while this one
    // runs) where that keeps the layout within 196 KB, the size above which
    // the SM's L1 carve-out halves (measured: the split query tiles with
    // two buffers at 32 rows, 224 KB, cost 13% on long contexts; one
    // buffer, 192 KB, 3.5%).
    static constexpr int QB = N <= (QSF == 2 ? 16 : 48) ? 2 : 1;
    // Tensor memory (512 columns): KB buffers of K codes (128 columns each),
    // two score buffers of N columns, then O^T in OB chunk buffers x two d
    // halves x N columns.  Two K buffers let the loaders write the K codes of
    // tile i+1 while the MMAs of tile i read tile i's; two O buffers let a
    // chunk's epilogue overlap the next chunk's first P.V.  Up to 32 rows
    // both fit; 48 and 64 rows keep two K buffers and one O (at 48 rows this
    // measured the same as one K and two O); 80 rows one K and one O.
    static constexpr int KB = N <= 64 ? 2 : 1;
    static constexpr int OB = N <= 32 ? 2 : 1;
    static constexpr uint32_t SW = (uint32_t)N;
    static constexpr uint32_t colS = 128u * KB;
    static constexpr uint32_t colO = colS + 2 * SW;
    static __device__ __forceinline__ uint32_t col_k(int kb) { return 128u * (uint32_t)kb; }
    static __device__ __forceinline__ uint32_t col_s(int par) { return colS + SW * (uint32_t)par; }
    static __device__ __forceinline__ uint32_t col_o(int cp, int hh)
    {
        return colO + 2 * SW * (uint32_t)(cp % OB) + SW * (uint32_t)hh;
    }
    static_assert(N % 16 == 0 && N <= kMaxRows, "MMA N");
    static_assert(colO + OB * 2 * SW <= kTmemCols, "tensor memory columns");
    static constexpr uint32_t v = 0;
    static constexpr uint32_t q = 2 * kStageBytes;
    static constexpr uint32_t pb = q + QB * N * 512u * QSF;
    static constexpr uint32_t misc = pb + PB * N * 256u;
    static constexpr uint32_t total = misc + (uint32_t)((sizeof(Misc) + 127) / 128 * 128);
};

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

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b)
{
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ---------------------------------------------------------------- work list

__device__ inline int seq_chunks(const Params &p, int b, int *start, int *n)
{
    seq_range(p, b, start, n);
    return *n > 0 ? (*n + p.chunk_cells - 1) / p.chunk_cells : 0;
}

// Quotient and remainder of non-negative a / b (b > 0): 32-bit division
// (a few instructions) whenever both fit, 64-bit otherwise.
__device__ __forceinline__ void divmod_nn(long long a, long long b, long long &q, long long &r)
{
    if (a < 0x7fffffffll && b < 0x7fffffffll) {
        const unsigned ua = (unsigned)a, ub = (unsigned)b;
        q = ua / ub;
        r = ua - (unsigned)q * ub;
    } else {
        q = a / b;
        r = a - q * b;
    }
}

// Position of the first item of CTA `cta` of `ncta` (the CTAs of one row
// block), computed by one full warp: lanes read the sequences' list offsets
// in parallel, a warp scan finds the sequence that holds item `lo`.  Items
// are (sequence, KV head, chunk) in that order; each CTA takes a contiguous
// range (consecutive chunks share their queries).
__device__ inline void cursor_init_warp(const Params &p, Cursor &cur, int lane, int cta, int ncta)
{
    cur.b = cur.g = cur.c = cur.nch = cur.start = cur.n = 0;
    cur.remaining = 0;
    cur.per = 1;
    cur.lo = 0;
    long long per, rem, q, r;
    if (p.sel_offsets == nullptr) {
        // one sequence (the step entry): closed form, no scan
        int s, n;
        const int nch = seq_chunks(p, 0, &s, &n);
        const long long total = (long long)p.G * nch;
        divmod_nn(total + ncta - 1, ncta, per, rem);
        const long long lo = per * cta;
        const long long hi = min(lo + per, total);
        if (lo >= hi) return;
        cur.remaining = (int)(hi - lo);
        cur.per = (int)per;
        cur.lo = lo;
        cur.nch = nch;
        cur.start = s;
        cur.n = n;
        divmod_nn(lo, nch, q, r);
        cur.g = (int)q;
        cur.c = (int)r;
        return;
    }
    long long total = 0;
    int s, n;
    for (int b = lane; b < p.n_seq; b += 32) total += (long long)p.G * seq_chunks(p, b, &s, &n);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    divmod_nn(total + ncta - 1, ncta, per, rem);
    const long long lo = per * cta;
    const long long hi = min(lo + per, total);
    if (lo >= hi) return;
    cur.remaining = (int)(hi - lo);
    cur.per = (int)per;
    cur.lo = lo;
    long long before = 0;
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
            divmod_nn(off, cur.nch, q, r);
            cur.g = (int)q;
            cur.c = (int)r;
            return;
        }
        before += __shfl_sync(0xffffffffu, incl, 31);
    }
    cur.remaining = 0;
}

__device__ __forceinline__ void cursor_next(const Params &p, Cursor &cur)
{
    if (--cur.remaining <= 0) return;
    if (++cur.c < cur.nch) return;
    cur.c = 0;
    if (++cur.g < p.G) return;
    cur.g = 0;
    // the next sequence with a non-empty list (the offsets were checked, and
    // any bad ones reported, when the CTA's first item was found)
    for (int b = cur.b + 1; b < p.n_seq; ++b) {
        const int o0 = __ldg(p.sel_offsets + b);
        const int n = min(__ldg(p.sel_offsets + b + 1) - o0, p.max_selected);
        if (o0 >= 0 && n > 0) {
            cur.b = b;
            cur.nch = (n + p.chunk_cells - 1) / p.chunk_cells;
            cur.start = o0;
            cur.n = n;
            return;
        }
    }
    cur.remaining = 0;
}

// First item of the next (sequence, KV head) pair in the range, if any.
__device__ inline Cursor next_segment(const Params &p, Cursor cur)
{
    const int left = cur.nch - 1 - cur.c; // later items of the same pair
    if (cur.remaining - 1 <= left) {
        cur.remaining = 0;
        return cur;
    }
    cur.remaining -= left;
    cur.c = cur.nch - 1;
    cursor_next(p, cur);
    return cur;
}

// The tile stream: every item's chunk in 128-cell tiles; a segment is a run
// of tiles of one (sequence, KV head) pair (one query block).
struct TileIt {
    Cursor cur;
    int ti, nt, nc; // tile within the chunk, tiles of the chunk, cells of the chunk
    int seg;
    bool valid;
};

__device__ __forceinline__ void tile_setup(const Params &p, TileIt &t)
{
    t.nc = min(p.chunk_cells, t.cur.n - t.cur.c * p.chunk_cells);
    t.nt = (t.nc + kTile - 1) / kTile;
    t.ti = 0;
}

__device__ __forceinline__ void tile_init(const Params &p, TileIt &t, const Cursor &first)
{
    t.cur = first;
    t.seg = 0;
    t.valid = first.remaining > 0;
    if (t.valid) tile_setup(p, t);
}

__device__ __forceinline__ void tile_next(const Params &p, TileIt &t)
{
    if (++t.ti < t.nt) return;
    const int b = t.cur.b, g = t.cur.g;
    cursor_next(p, t.cur);
    t.valid = t.cur.remaining > 0;
    if (!t.valid) return;
    tile_setup(p, t);
    if (t.cur.b != b || t.cur.g != g) ++t.seg;
}

__device__ __forceinline__ int tile_cells(const TileIt &t) { return min(kTile, t.nc - t.ti * kTile); }

__device__ __forceinline__ int tile_base(const Params &p, const TileIt &t)
{
    return t.cur.start + t.cur.c * p.chunk_cells + t.ti * kTile;
}

// First / last tile of a run (rem0: the CTA's item count; rem0 - remaining
// is the item's offset in the CTA's range).
__device__ __forceinline__ bool run_first(const TileIt &t, int rem0)
{
    return t.ti == 0 && (t.cur.c == 0 || (rem0 - t.cur.remaining) % kRunChunks == 0);
}

__device__ __forceinline__ bool run_last(const TileIt &t, int rem0)
{
    return t.ti == t.nt - 1 &&
           (t.cur.c == t.cur.nch - 1 || t.cur.remaining == 1 || (rem0 - t.cur.remaining + 1) % kRunChunks == 0);
}

// Items y in [0, n) whose offset in their CTA's range is a multiple of
// kRunChunks: full ranges of per items hold ceil(per / kRunChunks) each.
__device__ __forceinline__ long long run_starts_below(long long n, int per)
{
    long long q, r;
    divmod_nn(n, per, q, r);
    return q * ((per + kRunChunks - 1) / kRunChunks) + (r + kRunChunks - 1) / kRunChunks;
}

// Slot of the run that starts at item x, chunk c of its pair (the pair's
// first item is x - c, a run start whatever its offset), and the pair's run
// count.
__device__ __forceinline__ int run_slot(long long x, int c, int per)
{
    if (c == 0 || per == 1) return c; // (an item per CTA: a run per chunk)
    return (int)(1 + run_starts_below(x, per) - run_starts_below(x - c + 1, per));
}

__device__ __forceinline__ int run_count(long long pair0, int nch, int per)
{
    if (per == 1) return nch;
    return (int)(1 + run_starts_below(pair0 + nch, per) - run_starts_below(pair0 + 1, per));
}

// ---------------------------------------------------------------- step a1

constexpr int kBadPos = INT_MIN;

// Checked pool slot of a page entry `raw` and the position's offset in its
// page, -1 when masked or out of range; `report` raises the status bits (the
// one thread that resolves the cell reports).
__device__ __forceinline__ int slot_of(const Params &p, int raw, int off, bool report)
{
    if (raw == kBadPos) {
        if (report) raise_status(p, QSA_STATUS_BAD_POSITION);
        return -1;
    }
    if (raw == -1) return -1;
    if (raw < 0 || raw >= p.pool_pages) {
        if (report) raise_status(p, QSA_STATUS_BAD_SLOT);
        return -1;
    }
    return p.page_cells == 1 ? raw : raw * p.page_cells + off;
}

// ---------------------------------------------------------------- queries

// Element offset of query row r (= t*H + j) of (sequence b, KV head g).
__device__ __forceinline__ size_t q_row_offset(const Params &p, int b, int g, int r)
{
    const int t = r / p.H, j = r % p.H;
    return (((size_t)b * p.T + t) * p.G * p.H + (size_t)g * p.H + j) * kHeadDim;
}

// The K codes sit in tensor memory with the contraction index permuted (the
// loader's 16x256b stores, see the loader): tensor-memory dimension
// 16k + 4u + e holds byte (k < 8 ? 32u + 4k : 128 + 32u + 4(k - 8)) + e of
// the K row.  The query tile is stored in the same order, so the dot product
// is unchanged.  Piece pc (dimensions 8pc..8pc+7) of a query row takes the
// four elements at s0 and the four at s0 + 32.
__device__ __forceinline__ int q_piece_source(int pc)
{
    const int k = pc >> 1, u0 = (pc & 1) * 2;
    return (k < 8 ? 4 * k : 128 + 4 * (k - 8)) + 32 * u0;
}

// The raw elements of query piece pc of the row at `row`: four at s0 and
// four at s0 + 32 (f32: a and b whole; bf16: a.x, a.y and b.x, b.y).
struct QRaw {
    uint4 a, b;
};

__device__ __forceinline__ QRaw q_piece_load(const Params &p, const uint8_t *row, int pc)
{
    const int s0 = q_piece_source(pc);
    QRaw q;
    if (p.q_bf16) {
        const uint2 a = *reinterpret_cast<const uint2 *>(row + 2 * s0);
        const uint2 b = *reinterpret_cast<const uint2 *>(row + 2 * (s0 + 32));
        q.a = make_uint4(a.x, a.y, 0u, 0u);
        q.b = make_uint4(b.x, b.y, 0u, 0u);
    } else {
        q.a = *reinterpret_cast<const uint4 *>(row + 4 * s0);
        q.b = *reinterpret_cast<const uint4 *>(row + 4 * (s0 + 32));
    }
    return q;
}

// Raw query piece -> its f16 high parts hi and the f16 rounding lo of what
// they leave (q - hi is exact in fp32; bf16 elements are exact in f16, lo = 0).
__device__ __forceinline__ void q_piece_cvt2(const Params &p, const QRaw &q, uint4 &hi, uint4 &lo)
{
    float f[8];
    if (p.q_bf16) {
        f[0] = bf16_bits_to_f32(q.a.x & 0xffff); f[1] = bf16_bits_to_f32(q.a.x >> 16);
        f[2] = bf16_bits_to_f32(q.a.y & 0xffff); f[3] = bf16_bits_to_f32(q.a.y >> 16);
        f[4] = bf16_bits_to_f32(q.b.x & 0xffff); f[5] = bf16_bits_to_f32(q.b.x >> 16);
        f[6] = bf16_bits_to_f32(q.b.y & 0xffff); f[7] = bf16_bits_to_f32(q.b.y >> 16);
    } else {
        f[0] = __uint_as_float(q.a.x); f[1] = __uint_as_float(q.a.y);
        f[2] = __uint_as_float(q.a.z); f[3] = __uint_as_float(q.a.w);
        f[4] = __uint_as_float(q.b.x); f[5] = __uint_as_float(q.b.y);
        f[6] = __uint_as_float(q.b.z); f[7] = __uint_as_float(q.b.w);
    }
    float r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = f[i] - __half2float(__float2half_rn(f[i]));
    hi = make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]), pack_f16x2(f[6], f[7]));
    lo = make_uint4(pack_f16x2(r[0], r[1]), pack_f16x2(r[2], r[3]), pack_f16x2(r[4], r[5]), pack_f16x2(r[6], r[7]));
}

// Query tiles of every (sequence, KV head) pair, written once per call into
// the workspace in exactly the shared-memory layout the MMA reads (f16,
// K-major, 128-byte swizzle, contraction index permuted as above, rows >= R
// zero; the high parts, then the low parts where the layout has them), so
// the chunk kernel brings a pair's tile in with one bulk copy.  A thread
// converts 16-byte pieces (eight elements) of it.
template <int N>
__global__ void __launch_bounds__(128) qsa_query_stage_kernel(const Params p)
{
    // Launched as a programmatic dependent of the kernel before the call on
    // the stream (if any, the previous call's merge).  The chunk kernel may
    // launch at once: before it waits for this grid it only reads the
    // caller's inputs (list, page table, pools).  This kernel reads and
    // converts its pieces of the caller's queries, then waits for the kernel
    // before it, whose chunk kernel may still be reading the query images,
    // before it writes them; so once this grid is complete the call before
    // is too, and the chunk kernel's wait for it covers its partial writes as
    // well.  A grid of at most one 128-thread CTA per SM (each thread takes
    // pieces e, e + stride, ...), so the grid is soon resident and lets the
    // chunk kernel launch.
    cudaTriggerProgrammaticLaunchCompletion();
    // one image per (pair, row block): rows rb * rb_rows .. of the pair
    const int n_rb = p.row_blocks > 1 ? p.row_blocks : 1;
    const int rb_rows = n_rb > 1 ? p.rb_rows : p.R;
    const long long pieces = (long long)p.n_seq * p.G * n_rb * N * 32;
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long e0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    constexpr int QSF = Lay<N>::QSF;
    auto convert = [&](long long e, uint4 &v, uint4 &lo) {
        const int img_i = (int)(e / (N * 32));
        const int bg = img_i / n_rb, rblk = img_i % n_rb;
        const int r = (int)((e / 32) % N), pc = (int)(e % 32);
        const int row = rblk * rb_rows + r;
        v = make_uint4(0, 0, 0, 0);
        lo = make_uint4(0, 0, 0, 0);
        if (r < rb_rows && row < p.R) {
            const int esz = p.q_bf16 ? 2 : 4;
            q_piece_cvt2(p, q_piece_load(p, static_cast<const uint8_t *>(p.q) + q_row_offset(p, bg / p.G, bg % p.G, row) * esz, pc), v, lo);
        }
    };
    auto store = [&](long long e, const uint4 &v, const uint4 &lo) {
        const int img_i = (int)(e / (N * 32));
        const int r = (int)((e / 32) % N), pc = (int)(e % 32);
        uint8_t *img = static_cast<uint8_t *>(p.q_img) + (size_t)img_i * N * 512 * QSF + kmajor_sw128_off(r, pc * 8, N);
        *reinterpret_cast<uint4 *>(img) = v;
        if (QSF == 2) *reinterpret_cast<uint4 *>(img + N * 512) = lo;
    };
    constexpr int kEarly = 4; // pieces per thread converted before the wait
    uint4 hv[kEarly], lv[kEarly];
#pragma unroll
    for (int k = 0; k < kEarly; ++k)
        if (e0 + k * stride < pieces) convert(e0 + k * stride, hv[k], lv[k]);
    cudaGridDependencySynchronize();
#pragma unroll
    for (int k = 0; k < kEarly; ++k)
        if (e0 + k * stride < pieces) store(e0 + k * stride, hv[k], lv[k]);
    for (long long e = e0 + kEarly * stride; e < pieces; e += stride) {
        uint4 v, lo;
        convert(e, v, lo);
        store(e, v, lo);
    }
}

// ---------------------------------------------------------------- kernel

// N: MMA columns (rows padded to 16); KR: 8-row score blocks that hold real
// rows (KR * 8 >= R), the softmax skips the rest; LIM: the call carries
// causal limits per query (a separate instantiation, so calls without them
// run exactly the code they ran before limits existed).
template <int N, int KR, bool LIM>
__global__ void __launch_bounds__(kThreads, 1) qsa_chunk_tc_kernel(const Params p)
{
    using L = Lay<N>;
    constexpr int PB = L::PB;
    constexpr int NR = 2 * KR; // score rows a softmax thread holds: 8k + 2u + e
    // The operand tiles need 1024-byte alignment (128-byte swizzle atoms); the
    // dynamic shared memory of a kernel without static shared memory starts
    // there, so no padding is reserved (it would cost the 196 KB shared-memory
    // carve-out at 32 and 64 query columns).  The check keeps a misplaced
    // window from being used.
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) raise_status(p, QSA_STATUS_LAUNCH);
        return;
    }
    Misc &ms = *reinterpret_cast<Misc *>(smem + L::misc);
    const int tid = threadIdx.x;
    // the warp index read through a shuffle: provably the same in every
    // lane, so values derived from it (tensor-memory addresses, roles) stay
    // in uniform registers and warp-wide tcgen05 operations need no per-lane
    // fallback
    const int w = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
    // Row block: the CTAs of block rb take rows row0 .. row0 + Rl - 1 of every
    // item (all rows when the rows are not split).
    const int n_rb = p.row_blocks > 1 ? p.row_blocks : 1;
    const int cta_per_rb = (int)gridDim.x / n_rb;
    const int rblk = (int)blockIdx.x / cta_per_rb;
    const int row0 = n_rb > 1 ? rblk * p.rb_rows : 0;
    const int Rl = n_rb > 1 ? min(p.rb_rows, p.R - row0) : p.R;
    const uint32_t s_v = smem_u32(smem + L::v);
    const uint32_t s_q = smem_u32(smem + L::q);
    const uint32_t s_p = smem_u32(smem + L::pb);

    if (tid == 0) {
        mbar_init(&ms.s_done, 1);
        mbar_init(&ms.pv_done, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms.k_full[i], kLoadThreads);
            mbar_init(&ms.k_empty[i], 1);
            mbar_init(&ms.v_full[i], kLoadThreads);
            mbar_init(&ms.v_empty[i], 1);
            mbar_init(&ms.sc_full[i], kResolveThreads);
            mbar_init(&ms.sc_empty[i], kSoftThreads);
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.s_empty[i], kSoftThreads);
            mbar_init(&ms.p_full[i], kSoftThreads);
            mbar_init(&ms.p_empty[i], 1);
            mbar_init(&ms.o_full[i], 1);
            mbar_init(&ms.o_empty[i], kSoftThreads);
            // bulk copy (one arrival + bytes), or the softmax threads' stores
            mbar_init(&ms.q_full[i], p.q_inline ? kSoftThreads : 1);
            mbar_init(&ms.q_empty[i], 1);
        }
        for (int r = 0; r < kMaxRows + 4; ++r) ms.red_fac[r] = 1.f;
        ms.abort = 0;
        fence_mbar_init();
    }
    if (w == kMmaWarp) {
        tmem_alloc(&ms.tmem, kTmemCols);
        tmem_relinquish();
    }
    if (w == kLoadWarps) cursor_init_warp(p, ms.first, lane, (int)blockIdx.x - rblk * cta_per_rb, cta_per_rb);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the merge kernel may be scheduled now; it waits for this grid's results
    cudaTriggerProgrammaticLaunchCompletion();
    // (shuffled from lane 0 for the same reason as the warp index)
    const uint32_t tmem = __shfl_sync(0xffffffffu, ms.tmem, 0);
    Cursor first;
    first.b = __shfl_sync(0xffffffffu, ms.first.b, 0);
    first.g = __shfl_sync(0xffffffffu, ms.first.g, 0);
    first.c = __shfl_sync(0xffffffffu, ms.first.c, 0);
    first.nch = __shfl_sync(0xffffffffu, ms.first.nch, 0);
    first.start = __shfl_sync(0xffffffffu, ms.first.start, 0);
    first.n = __shfl_sync(0xffffffffu, ms.first.n, 0);
    first.remaining = __shfl_sync(0xffffffffu, ms.first.remaining, 0);

    // Waits: a completed phase costs one test.  Otherwise the thread
    // suspends between tests (for short bounds, used to exercise the
    // time-out path, it polls); a wait that runs out raises
    // QSA_STATUS_TIMEOUT and sets the CTA's abort flag, after which waits
    // return at once and the roles run to the end of their loops.
    volatile int *abort_flag = &ms.abort;
    const uint32_t suspend_ns = p.wait_cycles >= (1ll << 24) ? 200000u : 0u;
    auto wait = [&](uint64_t *bar, uint32_t parity) {
        if (mbar_test_wait(bar, parity) || *abort_flag) return;
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, parity, suspend_ns)) {
            if (clock64() - t0 > p.wait_cycles) {
                *abort_flag = 1;
                raise_status(p, QSA_STATUS_TIMEOUT);
                return;
            }
        }
    };

    if (w < kLoadWarps) {
        // ================================================================ loaders
        // Warp w covers the 16 tile rows (cells) R0 = 32(w%4) + 16(w/4) .. R0+15.
        // K: thread t holds cells A = R0 + t/4 and B = A + 8 and, of each, the
        // 32-byte pieces at bytes 32u and 128 + 32u (u = t%4): every warp load
        // reads 8 whole 128-byte lines, and the pieces land in tensor memory by
        // 16x256b stores (lanes t/4 and 8 + t/4, columns 8k + 2u, +1).
        // V: thread t holds cells A' = R0 + t%8 and B' = A' + 8, pieces at
        // 32v and 128 + 32v (v = t/8), so the 16-byte swizzled shared-memory
        // stores of 8 consecutive threads hit 8 different bank groups.
        const int R0 = 32 * (w & 3) + 16 * (w >> 2);
        const int u = lane & 3;
        const int vr = lane & 7, vu = lane >> 3, vA = R0 + vr; // and B' = A' + 8
        const bool res = lane < 16; // resolves cell R0 + lane, reports its status
        const int cr = R0 + (lane & 15);
        const uint32_t t_lane = (uint32_t)R0 << 16;
        // V stores: piece i of (cell A' + 8rr, 32 dims at byte 128pc + 32vu) goes
        // to d-block 2pc + vu/2, row group (A' + 8rr)/8, row A' % 8, 16-byte
        // chunk (4(vu&1) + i) ^ (A' % 8): a base plus rr * 1024 + pc * 32768
        // plus one of four swizzled chunk offsets
        const uint32_t vbase = (uint32_t)((vu >> 1) * 16384 + (vA >> 3) * 1024 + vr * 128);
        uint32_t vchunk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) vchunk[i] = (uint32_t)(((4 * (vu & 1) + i) ^ vr) << 4);
        // Resolution (step a1) runs ahead of the row loads through shared-memory
        // rings filled by 4-byte asynchronous copies, so no register waits on
        // those reads: step j copies the list entries of tile j+6, the page
        // entries of tile j+4 (from list entries copied two steps earlier),
        // checks the slots of tile j+2 (from page entries copied two steps
        // earlier), prefetches that tile's rows into L2 and copies its scales;
        // the rows of tile j+1 are loaded into registers; tile j is converted.
        // tile info per stage: bg = b * G + g, mt = cells of the tile (0 = none)
        int bg1 = 0, bg2 = 0, bg3 = 0, bg4 = 0, bg5 = 0, bg6 = 0;
        int sq4 = 0, sq5 = 0, sq6 = 0; // sequence of the tile at stages 4-6 (its page-table row)
        int mt0 = 0, mt1 = 0, mt2 = 0, mt3 = 0, mt4 = 0, mt5 = 0, mt6 = 0;
        // slots (-1: masked) of the K cells A, B and the V cells A', B' at stages 1 and 2
        int kA1 = -1, kB1 = -1, vA1 = -1, vB1 = -1, kA2 = -1, kB2 = -1, vA2 = -1, vB2 = -1;
        uint32_t rk[32], rv[32]; // K: A p0, A p1, B p0, B p1; V: A' p0, A' p1, B' p0, B' p1
#pragma unroll
        for (int e = 0; e < 32; ++e) rk[e] = rv[e] = 0u;
        TileIt head;
        tile_init(p, head, first);
        for (int j = -6;; ++j) {
            cp_async_wait_group<1>(); // the copies of step j-2 and earlier have landed
            // ---- tile j: K codes -> tensor memory
            if (mt0) {
                const int kb = j % L::KB;
                if (j >= L::KB) wait(&ms.k_empty[kb], (uint32_t)((j - L::KB) / L::KB) & 1u);
                tc_fence_after();
#pragma unroll
                for (int pc = 0; pc < 2; ++pc) {
#pragma unroll
                    for (int hq = 0; hq < 2; ++hq) {
                        uint32_t f[16];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            i8x4_to_f16x4(rk[8 * pc + 4 * hq + k], f[4 * k], f[4 * k + 1]);
                            i8x4_to_f16x4(rk[16 + 8 * pc + 4 * hq + k], f[4 * k + 2], f[4 * k + 3]);
                        }
                        tmem_st_16x256b_x4(tmem + t_lane + L::col_k(kb) + 64u * pc + 32u * hq, f);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&ms.k_full[kb]);
            } else if (j >= 0) {
                break;
            }
            // ---- rows of tile j+1 (K); a masked cell loads nothing (its score
            // is -inf and its probability 0 whatever the registers hold)
            const size_t kvb1 = (size_t)bg1 * p.pool_cells;
            if (mt1) {
                const int8_t *ka = p.k_pool + (kvb1 + (size_t)max(kA1, 0)) * kHeadDim + 32 * u;
                const int8_t *kb = p.k_pool + (kvb1 + (size_t)max(kB1, 0)) * kHeadDim + 32 * u;
                ldg256_stream_if(ka, rk, kA1 >= 0);
                ldg256_stream_if(ka + 128, rk + 8, kA1 >= 0);
                ldg256_stream_if(kb, rk + 16, kB1 >= 0);
                ldg256_stream_if(kb + 128, rk + 24, kB1 >= 0);
            }
            if (mt0) {
                const int jb = j & 1;
                if (res) {
                    // the scales and validity of tile j sit in ring entry j % 4
                    // (copied by this thread two steps ago); the softmax frees
                    // the entry of tile j-2, which the slot stage below reuses
                    if (j >= 2) wait(&ms.sc_empty[jb], (uint32_t)((j - 2) >> 1) & 1u);
                    if (LIM) ms.sc_r0[jb][cr] = ms.rs_r0[j & 3][cr];
                    mbar_arrive(&ms.sc_full[jb]);
                }
                // ---- tile j: V codes -> shared memory
                if (j >= 2) wait(&ms.v_empty[jb], (uint32_t)((j - 2) >> 1) & 1u);
                uint8_t *sv = smem + L::v + (size_t)jb * kStageBytes;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
                    for (int pc = 0; pc < 2; ++pc) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint4 v;
                            i8x4_to_f16x4(rv[16 * rr + 8 * pc + 2 * i], v.x, v.y);
                            i8x4_to_f16x4(rv[16 * rr + 8 * pc + 2 * i + 1], v.z, v.w);
                            *reinterpret_cast<uint4 *>(sv + vbase + (uint32_t)(rr * 1024 + pc * 32768) + vchunk[i]) = v;
                        }
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&ms.v_full[jb]);
            }
            // ---- rows of tile j+1 (V)
            if (mt1) {
                const int8_t *va = p.v_pool + (kvb1 + (size_t)max(vA1, 0)) * kHeadDim + 32 * vu;
                const int8_t *vb = p.v_pool + (kvb1 + (size_t)max(vB1, 0)) * kHeadDim + 32 * vu;
                ldg256_stream_if(va, rv, vA1 >= 0);
                ldg256_stream_if(va + 128, rv + 8, vA1 >= 0);
                ldg256_stream_if(vb, rv + 16, vB1 >= 0);
                ldg256_stream_if(vb + 128, rv + 24, vB1 >= 0);
            }
            // ---- list entries of tile j+6
            mt6 = 0;
            if (head.valid) {
                const int nc = tile_cells(head);
                bg6 = head.cur.b * p.G + head.cur.g;
                sq6 = head.cur.b;
                mt6 = nc;
                if (res && cr < nc) cp_async4(smem_u32(&ms.rs_sel[(j + 6) & 3][cr]), p.sel + tile_base(p, head) + cr);
                tile_next(p, head);
            }
            // ---- page-table entries of tile j+4 (from its list entries)
            if (mt4 && res) {
                const int e4 = (j + 4) & 3;
                int32_t *dst = &ms.rs_pg[e4][cr];
                if (cr >= mt4) {
                    *dst = -1; // past the tile's cells: masked
                } else {
                    // position pos: page pos / P, offset pos % P (P = 1: the entry is the slot)
                    const int pos = ms.rs_sel[e4][cr], P = p.page_cells;
                    const int32_t *prow = p.page_table + (size_t)sq4 * p.page_table_len;
                    if (LIM && pos >= 0) {
                        // rows t*H.. of the queries whose limit is above pos see the
                        // cell: with limits non-decreasing in t, those are the rows
                        // from H * #{t : limit[t] <= pos} on
                        const int32_t *lim = p.q_limit + (size_t)sq4 * p.T;
                        int below = 0;
                        for (int t = 0; t < p.T; ++t) below += __ldg(lim + t) <= pos;
                        ms.rs_r0[e4][cr] = (uint8_t)(below * p.H); // <= T * H <= 80
                    }
                    if (pos < 0 || (long long)pos >= (long long)p.page_table_len * P) {
                        *dst = kBadPos;
                    } else if (P == 1) {
                        cp_async4(smem_u32(dst), prow + pos);
                    } else {
                        const int page = pos / P;
                        ms.rs_off[e4][cr] = pos - page * P;
                        cp_async4(smem_u32(dst), prow + page);
                    }
                }
            }
            // ---- slots of tile j+2 (from its page entries): scales copied into
            // the ring, rows prefetched into L2
            if (mt2) {
                int sl = -1;
                if (res) {
                    const int e2 = (j + 2) & 3;
                    sl = slot_of(p, ms.rs_pg[e2][cr], ms.rs_off[e2][cr], true);
                    const size_t kvb = (size_t)bg2 * p.pool_cells;
                    if (sl >= 0) {
                        cp_async4(smem_u32(&ms.rs_ks[e2][cr]), p.k_scale + kvb + sl);
                        cp_async4(smem_u32(&ms.rs_vs[e2][cr]), p.v_scale + kvb + sl);
                    } else {
                        ms.rs_ks[e2][cr] = 0.f;
                        ms.rs_vs[e2][cr] = 0.f;
                    }
                    ms.rs_ok[e2][cr] = sl >= 0;
                }
                kA2 = __shfl_sync(0xffffffffu, sl, lane >> 2);
                kB2 = __shfl_sync(0xffffffffu, sl, (lane >> 2) + 8);
                vA2 = __shfl_sync(0xffffffffu, sl, vr);
                vB2 = __shfl_sync(0xffffffffu, sl, vr + 8);
                const int pf = __shfl_sync(0xffffffffu, sl, lane & 15); // cell R0 + lane%16, half lane/16
                if (pf >= 0) {
                    const size_t cell = (size_t)bg2 * p.pool_cells + pf;
                    prefetch_l2(p.k_pool + cell * kHeadDim + 128 * (lane >> 4));
                    prefetch_l2(p.v_pool + cell * kHeadDim + 128 * (lane >> 4));
                }
            }
            cp_async_commit();
            // shift the pipeline by one tile
            bg1 = bg2; bg2 = bg3; bg3 = bg4; bg4 = bg5; bg5 = bg6;
            sq4 = sq5; sq5 = sq6;
            mt0 = mt1; mt1 = mt2; mt2 = mt3; mt3 = mt4; mt4 = mt5; mt5 = mt6;
            kA1 = kA2; kB1 = kB2; vA1 = vA2; vB1 = vB2;
        }
        cp_async_wait_group<0>();
    } else if (w < kMmaWarp) {
        // ================================================================ softmax
        const int q = w & 3, c = 32 * q + lane;
        const int u = lane & 3, ra = lane >> 2; // 16x256b: rows 8k + 2u + e, cells 32q + 8i + ra
        const int orow = 4 * lane + q;          // the row this thread writes at a chunk's end
        constexpr int NK = N / 8;               // 16x256b repetitions over the score columns
        const uint32_t t_lane = (uint32_t)(32 * q) << 16;
        struct Pend {
            int b, g, k, cp, runs; // partial slot k; the pair's run count when k == 0
            bool on;
        };
        Pend pend{0, 0, 0, 0, 0, false};
        int run_k = 0, run_n = 0; // slot of the current run; its pair's run count (slot 0)
        // per row (index 2k + e = row 8k + 2u + e): the reference maximum (log2
        // units, the same in every thread that holds the row; -FLT_MAX until
        // the row's first valid score, when all its scores are -inf), and this
        // thread's share of the chunk's sum of probabilities and of its maximum
        float mref[NR], lsum[NR], cmax[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            mref[r] = -FLT_MAX;
            lsum[r] = 0.f;
            cmax[r] = -INFINITY;
        }
        float sig = 0.f, inv_sig = 0.f; // the V-scale reference of the pair, 0 before its first cell
        int cp = -1, cur_seg = -1;
        TileIt it;
        tile_init(p, it, first);

        // partials of chunk e.cp: O read out of tensor memory, times sigma * 2^(mref - m)
        // The call before may still be reading the workspace (the partials):
        // a single-pair call waits for it just before its first partial
        // store, so its first tile runs under the previous call's merge.
        // (The softmax threads store nothing else to global memory; with
        // staged queries the S warp's wait for the staging grid, which
        // waited for the call before, comes first.)
        bool prev_done = !p.q_inline;

        // partials of run e.cp: O read out of tensor memory, times sigma *
        // 2^(mref - m), and the m and l that the run's end left in shared memory
        auto epilogue = [&](const Pend &e) {
            wait(&ms.o_full[e.cp % L::OB], (uint32_t)(e.cp / L::OB) & 1u);
            tc_fence_after();
            const size_t base = (((size_t)e.b * p.G + e.g) * p.n_chunks + e.k) * p.R + row0;
            const float *fin = ms.st_fin[e.cp & 1];
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                // all 8-row blocks that hold real rows in flight together, one wait
                float v[8 * KR];
#pragma unroll
                for (int k = 0; k < KR; ++k)
                    tmem_ld8(tmem + t_lane + L::col_o(e.cp, hh) + 8u * k, v + 8 * k);
                tmem_wait_ld();
                regs_after_wait<8 * KR>(v);
                if (!prev_done) {
                    cudaGridDependencySynchronize();
                    prev_done = true;
                }
                float *dst = p.part_o + base * kHeadDim + 128 * hh + c;
#pragma unroll
                for (int k = 0; k < KR; ++k) {
                    const float4 f0 = *reinterpret_cast<const float4 *>(fin + 8 * k);
                    const float4 f1 = *reinterpret_cast<const float4 *>(fin + 8 * k + 4);
                    const float fr[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int r = 8 * k + jj; // rows R..N-1 are MMA padding
                        if (r < Rl) dst[(size_t)r * kHeadDim] = v[r] * fr[jj];
                    }
                }
            }
            if (c < Rl) {
                p.part_m[base + c] = ms.st_m[e.cp & 1][c];
                p.part_l[base + c] = ms.st_l[e.cp & 1][c];
            }
            if (e.k == 0 && c == 0 && rblk == 0) p.part_runs[(size_t)e.b * p.G + e.g] = e.runs;
            tc_fence_before();
            mbar_arrive(&ms.o_empty[e.cp % L::OB]);
        };

        // end of run cp: the rows' true maxima and sums across the CTA; the
        // row's owner leaves m, l and the factor its O is read out with in
        // shared memory for the epilogue
        auto run_end = [&](int chunk) {
            const int cpar = chunk & 1;
            float cm[NR], cs[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                cm[r] = cmax[r];
                cs[r] = lsum[r];
            }
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    cm[r] = fmaxf(cm[r], __shfl_xor_sync(0xffffffffu, cm[r], o));
                    cs[r] += __shfl_xor_sync(0xffffffffu, cs[r], o);
                }
            }
#pragma unroll
            for (int k = 0; k < KR; ++k) {
                if (ra == (k & 7)) {
                    *reinterpret_cast<float2 *>(&ms.ch_max[q][8 * k + 2 * u]) = make_float2(cm[2 * k], cm[2 * k + 1]);
                    *reinterpret_cast<float2 *>(&ms.ch_sum[q][8 * k + 2 * u]) = make_float2(cs[2 * k], cs[2 * k + 1]);
                    if (q == 0)
                        *reinterpret_cast<float2 *>(&ms.ch_ref[8 * k + 2 * u]) = make_float2(mref[2 * k], mref[2 * k + 1]);
                }
            }
            named_bar(kBarSoft, kSoftThreads);
            if (orow < Rl) {
                const float m = fmaxf(fmaxf(ms.ch_max[0][orow], ms.ch_max[1][orow]),
                                      fmaxf(ms.ch_max[2][orow], ms.ch_max[3][orow]));
                const float l = ((ms.ch_sum[0][orow] + ms.ch_sum[1][orow]) + ms.ch_sum[2][orow]) +
                                ms.ch_sum[3][orow];
                // (a row with a valid score has a finite reference)
                const float fin = m > -INFINITY ? fast_exp2(ms.ch_ref[orow] - m) : 0.f;
                ms.st_fin[cpar][orow] = fin * sig;
                ms.st_m[cpar][orow] = m > -INFINITY ? m * kLn2 : -INFINITY;
                ms.st_l[cpar][orow] = l * fin;
            }
        };

        if (p.q_inline && it.valid) {
            // One (sequence, KV head) in the whole call: this CTA converts its
            // rows of the query tile itself into buffer 0, in the layout of
            // the staged images (f16 high and low parts, K-major, 128-byte
            // swizzle, permuted contraction index, rows past its block zero),
            // while the loaders resolve the first tiles.  Nothing of the
            // previous call is read or written here.
            const int esz = p.q_bf16 ? 2 : 4;
            for (int e = c; e < N * 32; e += kSoftThreads) {
                const int r = e >> 5, pc = e & 31;
                uint4 v = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
                if (r < Rl) q_piece_cvt2(p, q_piece_load(p, static_cast<const uint8_t *>(p.q) + q_row_offset(p, first.b, first.g, row0 + r) * esz, pc), v, lo);
                *reinterpret_cast<uint4 *>(smem + L::q + kmajor_sw128_off(r, pc * 8, N)) = v;
                if (L::QSF == 2) *reinterpret_cast<uint4 *>(smem + L::q + N * 512 + kmajor_sw128_off(r, pc * 8, N)) = lo;
            }
            fence_proxy_async_smem();
            mbar_arrive(&ms.q_full[0]);
        }

        const int rem0 = first.remaining;
        for (int i = 0; it.valid; ++i) {
            const int par = i & 1;
            // first / last tile of a run (O, the row sums and maxima start
            // afresh at a run's first tile; its partials go out after the last)
            const bool first_t = run_first(it, rem0), last_t = run_last(it, rem0);
            if (it.seg != cur_seg) { // new (sequence, KV head): new rows, no reference yet
                cur_seg = it.seg;
#pragma unroll
                for (int r = 0; r < NR; ++r) mref[r] = -FLT_MAX;
                sig = inv_sig = 0.f;
            }
            if (first_t) {
                ++cp;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    lsum[r] = 0.f;
                    cmax[r] = -INFINITY;
                }
                const long long x = ms.first.lo + (rem0 - it.cur.remaining);
                run_k = run_slot(x, it.cur.c, ms.first.per);
                run_n = run_k == 0 ? run_count(x - it.cur.c, it.cur.nch, ms.first.per) : 0;
            }
            wait(&ms.sc_full[par], (uint32_t)(i >> 1) & 1u);
            // this thread's four cells (16x256b layout): cell(ci) = 32q + 8ci + t/4,
            // ci = 2L + B for lane group L (lanes +16) and row half B (+8)
            // per cell: K scale (x softmax scale x log2 e), V scale (0 when the
            // cell is masked), and a bias of -inf that masks the cell's scores
            float ksc[4], vsc[4], kbias[4];
            int r0[4]; // causal limits: the cell's first visible query row
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
                const int cc = 32 * q + 8 * ci + ra;
                kbias[ci] = ms.rs_ok[i & 3][cc] != 0 ? 0.f : -INFINITY;
                ksc[ci] = ms.rs_ks[i & 3][cc] * p.scale_log2;
                vsc[ci] = ms.rs_vs[i & 3][cc];
                r0[ci] = LIM ? ms.sc_r0[par][cc] : 0;
            }
            mbar_arrive(&ms.sc_empty[par]);
            wait(&ms.s_full[par], (uint32_t)(i >> 1) & 1u);
            tc_fence_after();
            // scores: x[L][4k + 2B + e] = cell 2L+B, row 8k + 2u + e (log2 units)
            float x[2][4 * NK];
            tmem_ld_16x256b<NK>(tmem + ((uint32_t)(32 * q) << 16) + L::col_s(par), x[0]);
            tmem_ld_16x256b<NK>(tmem + ((uint32_t)(32 * q + 16) << 16) + L::col_s(par), x[1]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&ms.s_empty[par]); // the scores live in registers from here on
            // ---- scale and mask; the vote: does a score pass its row's
            // reference by more than 2^8, or a V scale sigma by 16x (the first
            // valid cell of a pair passes both)?  The same rounded product is
            // used for the probabilities, so the max cell gets exactly 2^0.
            bool need = false;
#pragma unroll
            for (int k = 0; k < KR; ++k) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float m = -INFINITY;
#pragma unroll
                    for (int L2 = 0; L2 < 2; ++L2) {
#pragma unroll
                        for (int B = 0; B < 2; ++B) {
                            const int ci = 2 * L2 + B;
                            float &xv = x[L2][4 * k + 2 * B + e];
                            xv = __fmaf_rn(xv, ksc[ci], kbias[ci]); // = the rounded product, or -inf
                            if (LIM && row0 + 8 * k + 2 * u + e < r0[ci]) xv = -INFINITY; // beyond its query's limit
                            m = fmaxf(m, xv);
                        }
                    }
                    cmax[2 * k + e] = fmaxf(cmax[2 * k + e], m);
                    need |= m > mref[2 * k + e] + kRescaleLog2;
                }
            }
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) need |= fabsf(vsc[ci]) > sig * kSigmaGrow;
            if (named_bar_or(kBarSoft, kSoftThreads, need)) {
                // ---- the tile's true row maxima and largest V scale (rare: the
                // first tile of a pair, or a jump of 2^8)
                float tm[NR];
#pragma unroll
                for (int k = 0; k < KR; ++k)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        tm[2 * k + e] = fmaxf(fmaxf(x[0][4 * k + e], x[0][4 * k + 2 + e]),
                                              fmaxf(x[1][4 * k + e], x[1][4 * k + 2 + e]));
#pragma unroll
                for (int o = 4; o <= 16; o <<= 1)
#pragma unroll
                    for (int r = 0; r < NR; ++r) tm[r] = fmaxf(tm[r], __shfl_xor_sync(0xffffffffu, tm[r], o));
#pragma unroll
                for (int k = 0; k < KR; ++k)
                    if (ra == (k & 7))
                        *reinterpret_cast<float2 *>(&ms.red_max[q][8 * k + 2 * u]) = make_float2(tm[2 * k], tm[2 * k + 1]);
                {
                    float va = 0.f;
#pragma unroll
                    for (int ci = 0; ci < 4; ++ci) va = fmaxf(va, fabsf(vsc[ci])); // (0 if masked)
                    const unsigned uu = __reduce_max_sync(0xffffffffu, __float_as_uint(va));
                    if (lane == 0) ms.red_max[q][kMaxRows] = __uint_as_float(uu);
                }
                named_bar(kBarSoft, kSoftThreads);
                // every thread takes the same decisions for the rows it holds;
                // O of this run (if any is accumulated) is rescaled by rows
                bool resc = false;
#pragma unroll
                for (int k = 0; k < KR; ++k) {
                    float2 t2 = *reinterpret_cast<const float2 *>(&ms.red_max[0][8 * k + 2 * u]);
#pragma unroll
                    for (int ww = 1; ww < 4; ++ww) {
                        const float2 o2 = *reinterpret_cast<const float2 *>(&ms.red_max[ww][8 * k + 2 * u]);
                        t2.x = fmaxf(t2.x, o2.x);
                        t2.y = fmaxf(t2.y, o2.y);
                    }
                    float fac[2] = {1.f, 1.f};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int r = 2 * k + e;
                        const float t = e ? t2.y : t2.x;
                        if (t > mref[r] + kRescaleLog2) {
                            if (mref[r] > -FLT_MAX) fac[e] = fast_exp2(mref[r] - t);
                            lsum[r] *= fac[e];
                            mref[r] = t;
                        }
                    }
                    if (!first_t && (fac[0] != 1.f || fac[1] != 1.f)) resc = true;
                    if (q == 0 && ra == (k & 7))
                        *reinterpret_cast<float2 *>(&ms.red_fac[8 * k + 2 * u]) = make_float2(fac[0], fac[1]);
                }
                const float st = fmaxf(fmaxf(ms.red_max[0][kMaxRows], ms.red_max[1][kMaxRows]),
                                       fmaxf(ms.red_max[2][kMaxRows], ms.red_max[3][kMaxRows]));
                float fs = 1.f;
                if (st > sig * kSigmaGrow) {
                    if (sig > 0.f && !first_t) {
                        fs = sig / st;
                        resc = true;
                    }
                    sig = st;
                    inv_sig = 1.f / st;
                }
                if (named_bar_or(kBarSoft, kSoftThreads, resc)) {
                    // P.V of the previous tile (same run) must be done
                    if (PB == 2) wait(&ms.p_empty[(i - 1) & 1], (uint32_t)((i - 1) >> 1) & 1u);
                    else wait(&ms.p_empty[0], (uint32_t)(i - 1) & 1u);
                    tc_fence_after();
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll 1
                        for (int rb = 0; rb < Rl; rb += 16) {
                            const uint32_t ta = tmem + t_lane + L::col_o(cp, hh) + rb;
                            float v[16];
                            tmem_ld16(ta, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) v[jj] *= ms.red_fac[rb + jj] * fs;
                            tmem_st16(ta, v);
                        }
                    }
                    tmem_wait_st();
                }
            }
            const int pbi = i % PB;
            if (i >= PB) wait(&ms.p_empty[pbi], (uint32_t)((i - PB) / PB) & 1u);
            uint8_t *p_tile = smem + L::pb + (size_t)pbi * N * 256;
            // ---- P' = f16(p * v_scale / sigma) into the B operand of the P.V
            // MMA (K-major [rows][cells]); this thread's share of the row sums
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
                const int cc = 32 * q + 8 * ci + ra;
                const float vsn = vsc[ci] * inv_sig; // 0 for a masked cell
                const int L2 = ci >> 1, B = ci & 1;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    // element (row 8k + 2u + e, cell cc) at pe + 1024k
                    const int r7 = 2 * u + e;
                    uint8_t *pe = p_tile + (cc >> 6) * N * 128 + r7 * 128 + ((((cc & 63) >> 3) ^ r7) << 4) + (cc & 7) * 2;
#pragma unroll
                    for (int k = 0; k < KR; ++k) {
                        const float pr = fast_exp2(x[L2][4 * k + 2 * B + e] - mref[2 * k + e]); // 0 if masked
                        lsum[2 * k + e] += pr;
                        *reinterpret_cast<__half *>(pe + 1024 * k) = __float2half_rn(pr * vsn);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&ms.p_full[pbi]);
            if (pend.on) {
                epilogue(pend);
                pend.on = false;
            }
            if (last_t) {
                run_end(cp);
                pend = Pend{it.cur.b, it.cur.g, run_k, cp, run_n, true};
            }
            tile_next(p, it);
        }
        if (pend.on) {
            named_bar(kBarSoft, kSoftThreads); // the owners' factors are written
            epilogue(pend);
        }
    } else if (w == kMmaWarp) {
        // ================================================================ S warp
        // All 32 lanes run the loop (so every value is warp-uniform); one
        // elected lane issues the MMAs, commits and query copies.
        const bool leader = elect_one();
        const uint32_t idesc_s = idesc_f16(128, N, false, false, false, false);
        TileIt it;
        tile_init(p, it, first);
        // query tiles: one bulk copy per segment into buffer seg % QB.  With
        // two buffers, the first two now and segment s + 1 once segment s
        // has started (its buffer was segment s - 1's, free after that
        // segment's last QK); with one, segment s + 1 after segment s ends.
        constexpr int QB = L::QB;
        int q_issued[2] = {0, 0}; // bulk copies issued into each buffer
        auto load_q = [&](const Cursor &sc, int seg) {
            const uint32_t bytes = (uint32_t)N * 512u * L::QSF;
            if (leader) {
                mbar_arrive_expect_tx(&ms.q_full[seg % QB], bytes);
                bulk_g2s(smem + L::q + (size_t)(seg % QB) * N * 512 * L::QSF,
                         static_cast<const uint8_t *>(p.q_img) +
                             (((size_t)sc.b * p.G + sc.g) * n_rb + rblk) * N * 512 * L::QSF, bytes,
                         &ms.q_full[seg % QB]);
            }
            ++q_issued[seg % QB];
        };
        Cursor qnext = first;
        int qseg = 0; // next segment whose tile is to be loaded
        if (it.valid && !p.q_inline) {
            cudaGridDependencySynchronize(); // the tiles come from the staging kernel
            for (; qseg < QB && qnext.remaining > 0; ++qseg) {
                load_q(qnext, qseg);
                qnext = next_segment(p, qnext);
            }
        }
        int cur_seg = -1;
        for (int i = 0; it.valid; ++i) {
            const int seg = it.seg;
            const bool seg_start = seg != cur_seg;
            if (seg_start) wait(&ms.q_full[seg % QB], (uint32_t)(seg / QB) & 1u);
            cur_seg = seg;
            const int kb = i % L::KB;
            wait(&ms.k_full[kb], (uint32_t)(i / L::KB) & 1u);
            if (i >= 2) wait(&ms.s_empty[i & 1], (uint32_t)((i - 2) >> 1) & 1u);
            tc_fence_after();
            const uint64_t qd0 = smem_desc(s_q + (uint32_t)(seg % QB) * N * 512u * L::QSF, 16, 1024);
            const uint32_t sd = tmem + L::col_s(i & 1);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint64_t bd = qd0 + (uint64_t)(((uint32_t)(kk >> 2) * N * 128u + (uint32_t)(kk & 3) * 32u) >> 4);
                    mma_f16_ts(sd, tmem + L::col_k(kb) + 8u * kk, bd, idesc_s, kk > 0 ? 1u : 0u);
                    if (L::QSF == 2)
                        mma_f16_ts(sd, tmem + L::col_k(kb) + 8u * kk, bd + (uint64_t)((N * 512u) >> 4), idesc_s, 1u);
                }
                mma_commit(&ms.k_empty[kb]);
                mma_commit(&ms.s_full[i & 1]);
            }
            __syncwarp();
            tile_next(p, it);
            const bool seg_end = !it.valid || it.seg != seg;
            if (seg_end && leader) mma_commit(&ms.q_empty[seg % QB]);
            if (QB == 2 && seg_start && seg >= 1 && qnext.remaining > 0) {
                wait(&ms.q_empty[(seg - 1) & 1], (uint32_t)((seg - 1) >> 1) & 1u);
                load_q(qnext, qseg);
                ++qseg;
                qnext = next_segment(p, qnext);
            }
            if (QB == 1 && seg_end && qnext.remaining > 0) {
                wait(&ms.q_empty[0], (uint32_t)seg & 1u);
                load_q(qnext, qseg);
                ++qseg;
                qnext = next_segment(p, qnext);
            }
        }
        // before the CTA leaves (also after a time-out): every MMA of this
        // warp complete, every query copy landed.  The k-th copy into a
        // buffer completes phase k - 1 of its barrier, which nothing else
        // arrives on.
        if (leader) mma_commit(&ms.s_done);
        __syncwarp();
        mbar_wait(&ms.s_done, 0, kDrainCycles);
        if (!p.q_inline)
            for (int bq = 0; bq < QB; ++bq)
                if (q_issued[bq] > 0) mbar_wait(&ms.q_full[bq], (uint32_t)(q_issued[bq] - 1) & 1u, kDrainCycles);
    } else {
        // ================================================================ P.V warp
        // A second issuing warp: one thread issues a tcgen05.mma every ~50-70
        // cycles on this GPU, so S of the next tile and P.V of the current one
        // go out from two warps side by side.  All lanes run the loop; one
        // elected lane issues.
        const bool leader = elect_one();
        const uint32_t idesc_o = idesc_f16(128, N, false, false, true, false);
        TileIt it;
        tile_init(p, it, first);
        int cp = -1;
        const int rem0 = first.remaining;
        for (int i = 0; it.valid; ++i) {
            const bool first_t = run_first(it, rem0), last_t = run_last(it, rem0); // of a run
            if (first_t) ++cp;
            wait(&ms.p_full[i % PB], (uint32_t)(i / PB) & 1u);
            wait(&ms.v_full[i & 1], (uint32_t)(i >> 1) & 1u);
            if (first_t && cp >= L::OB) wait(&ms.o_empty[cp % L::OB], (uint32_t)((cp - L::OB) / L::OB) & 1u);
            tc_fence_after();
            // descriptors built once; a K step only moves the start address
            // (field [0,14) in 16-byte units, no carry for shared addresses)
            const uint64_t ad0 = smem_desc(s_v + (uint32_t)(i & 1) * kStageBytes, 16384, 1024);
            const uint64_t bd0 = smem_desc(s_p + (uint32_t)(i % PB) * N * 256u, 16, 1024);
            const uint32_t d0 = tmem + L::col_o(cp, 0);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    // the two d halves interleaved: independent accumulators
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint64_t ad = ad0 + (uint64_t)(((uint32_t)(2 * hh) * 16384u + (uint32_t)kk * 2048u) >> 4);
                        const uint64_t bd = bd0 + (uint64_t)(((uint32_t)(kk >> 2) * N * 128u + (uint32_t)(kk & 3) * 32u) >> 4);
                        mma_f16_ss(d0 + L::SW * hh, ad, bd, idesc_o, (first_t && kk == 0) ? 0u : 1u);
                    }
                }
                mma_commit(&ms.v_empty[i & 1]);
                mma_commit(&ms.p_empty[i % PB]);
                if (last_t) mma_commit(&ms.o_full[cp % L::OB]);
            }
            __syncwarp();
            tile_next(p, it);
        }
        if (leader) mma_commit(&ms.pv_done);
        __syncwarp();
        mbar_wait(&ms.pv_done, 0, kDrainCycles);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int N, int KR, bool LIM = false>
cudaError_t launch_n(Params &p, cudaStream_t stream)
{
    int dev = 0, sms = 0, max_smem = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    static_assert(Lay<N>::total <= 232448, "shared memory of the chunk kernel");
    const uint32_t bytes = Lay<N>::total;
    if ((int)bytes > max_smem) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(qsa_chunk_tc_kernel<N, KR, LIM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)bytes)) != cudaSuccess)
        return e;
    const long long pieces = (long long)p.n_seq * p.G * (p.row_blocks > 1 ? p.row_blocks : 1) * N * 32;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (!p.q_inline) {
        cudaLaunchConfig_t scfg = {};
        const long long blocks = (pieces + 127) / 128;
        scfg.gridDim = dim3((unsigned)(blocks < sms ? blocks : sms));
        scfg.blockDim = dim3(128);
        scfg.stream = stream;
        scfg.attrs = attr;
        scfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&scfg, qsa_query_stage_kernel<N>, p)) != cudaSuccess) return e;
    }
    // one persistent CTA per SM at most; with split rows, each row block gets
    // the same number of CTAs
    const long long items = (long long)p.n_seq * p.G * p.n_chunks;
    const int n_rb = p.row_blocks > 1 ? p.row_blocks : 1;
    const long long per_rb = items < sms / n_rb ? items : sms / n_rb;
    if (per_rb < 1) return cudaErrorInvalidConfiguration;
    // items per CTA when every list is full (the kernel's count is at most
    // this): above one, CTAs combine runs of chunks and the merge reads the
    // run counts; its CTA shape follows the slots a row then has
    const long long per = (items + per_rb - 1) / per_rb;
    const long long run = per < kRunChunks ? per : kRunChunks;
    p.runs = per > 1 ? 1 : 0;
    p.merge_slots = (int)(per > 1 ? std::min<long long>(p.n_chunks, (p.n_chunks + run - 1) / run + 1) : p.n_chunks);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(per_rb * n_rb));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qsa_chunk_tc_kernel<N, KR, LIM>, p);
}

} // namespace

size_t chunk_tc_query_image_bytes(int n_seq, int G, int R)
{
    // the rows of a pair in row blocks of up to 64 rows, each padded to its
    // MMA N: at most N + 48 padded rows in all
    const size_t N = (size_t)(R + 15) / 16 * 16;
    return (size_t)n_seq * G * (N + 48) * 512 * 2;
}

cudaError_t launch_chunk_tc(Params &p, cudaStream_t stream)
{
    if (p.n_chunks == 0) return cudaSuccess;
    // one (sequence, KV head): every CTA works on the same query tile and
    // converts it itself, so the call is two kernels (chunk, merge)
    p.q_inline = p.n_seq * p.G == 1 ? 1 : 0;
    p.row_blocks = 1;
    p.rb_rows = p.R;
    if (p.q_inline && !p.q_limit) {
        // Few chunks on one query tile (a decode window of one sequence):
        // the SMs the chunks leave idle take blocks of the rows instead, so
        // each CTA's chain of softmax, P' and epilogue work covers fewer
        // rows.  Each block re-reads the chunk's cells (from L2, mostly).
        // Blocks of the smallest multiple of 16 rows such that the call's
        // CTAs take at most half the SMs: back to back, a call's CTAs start
        // under the previous call's (and its merge's), and CTAs beyond the
        // free SMs would start only when those end (measured, 2,051 cells:
        // 8-row blocks on 85 and 102 CTAs for 36 and 48 rows, 6.63 and 6.75
        // us per call; 16-row blocks on 51 CTAs, 6.20 and 6.15 us).  Blocks
        // of 16 rows also keep windows of 12 to 64 rows on one instantiation
        // (N = 16, two 8-row score blocks), so a run of calls with different
        // window sizes does not alternate kernels (8-row blocks up to 24 rows
        // beside 16-row ones above: 6.42 us per call over windows of 1-4
        // queries; one instantiation: 5.68).
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        for (int rb = 16; rb < p.R; rb += 16) {
            const int n_rb = (p.R + rb - 1) / rb;
            if ((long long)p.n_chunks * n_rb <= sms / 2) {
                p.row_blocks = n_rb;
                p.rb_rows = rb;
                switch (rb) {
                case 16: return launch_n<16, 2>(p, stream);
                case 32: return launch_n<32, 4>(p, stream);
                case 48: return launch_n<48, 6>(p, stream);
                default: return launch_n<64, 8>(p, stream);
                }
            }
        }
    }
    if (!p.q_inline && !p.q_limit && p.R > 24) {
        // Calls over several pairs with more than 24 rows: blocks of 24 rows
        // (MMA N = 32), each with its own CTAs and query images.  The softmax
        // warps' per-tile chain grows with the rows while the loaders' work
        // does not, and with 48 rows it set the pace (16 sequences x 2 KV
        // heads x 48 rows, one-tile chunks: 35.9 -> 30.5 us per call on
        // GB300; blocks of 16 rows, 34.3).  Each block re-reads the cells.
        p.row_blocks = (p.R + 23) / 24;
        p.rb_rows = 24;
        return launch_n<32, 3>(p, stream);
    }
    if (p.q_limit) { // causal limits: one instantiation per N (padding rows cost a little)
        switch ((p.R + 15) / 16) {
        case 1: return launch_n<16, 2, true>(p, stream);
        case 2: return launch_n<32, 4, true>(p, stream);
        case 3: return launch_n<48, 6, true>(p, stream);
        case 4: return launch_n<64, 8, true>(p, stream);
        case 5: return launch_n<80, 10, true>(p, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    switch ((p.R + 7) / 8) { // 8-row blocks of real rows; N = that, padded to 16
    case 1: return launch_n<16, 1>(p, stream);
    case 2: return launch_n<16, 2>(p, stream);
    case 3: return launch_n<32, 3>(p, stream);
    case 4: return launch_n<32, 4>(p, stream);
    case 5: return launch_n<48, 5>(p, stream);
    case 6: return launch_n<48, 6>(p, stream);
    case 7: return launch_n<64, 7>(p, stream);
    case 8: return launch_n<64, 8>(p, stream);
    case 9: return launch_n<80, 9>(p, stream);
    case 10: return launch_n<80, 10>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace qsa
