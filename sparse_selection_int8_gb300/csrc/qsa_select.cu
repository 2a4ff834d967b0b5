// qsa_select.cu -- QSA block selection: the scorer over pooled keys and its
// top-k, which produce the selected-cell list the decode attention reads.
//
// The step is the QSA selection scorer of "Strata issue #8, round 9:
// performance candidate set on v0.2.9" (R9-gpu-9: qsa_block_scores_rows over
// pooled keys, a dead tail, per-query indexer vectors and steps) followed by
// the top-k (the long-context select and TOPK_SPLIT of the same page's
// "Absorbed, considered and dropped" list).  The pages print no formula; the
// reading implemented here:
//   block j of a sequence covers positions [jR, (j+1)R) and has one pooled
//   key of F = idx_heads * idx_dim bf16 values; it is live while
//   jR < n_live, and a candidate for query t if also jR <= steps[t];
//   score s[t][j] = sum_f q_idx[t][f] * pooled[j][f] (-inf off candidates);
//   each query keeps its top_k candidates (ties to the lower block id);
//   the list is the union over the window's queries, expanded to the live
//   positions of the kept blocks in ascending order (CSR over sequences).
//
// Three launches on the stream (the second and third programmatic
// dependents of the one before, so each launches while its predecessor runs
// and waits for it before it reads its results):
//   scores   two blocks per warp, both pooled keys loaded before either is
//            used (16-byte loads), the queries from shared memory, a warp
//            butterfly per query; dead and future blocks read nothing
//   top-k    one CTA per (sequence, query): an exact four-pass radix select
//            over order-preserving 32-bit keys of the scores (shared memory;
//            a warp's histogram adds aggregated per digit), ties ranked by
//            block id with a block scan; kept ids ascending, their bits OR-ed
//            into the sequence's block bitmap.  The last of a sequence's CTAs
//            counts its positions per bitmap word; the last sequence counted
//            scans the sequences into the CSR offsets.
//   expand   one warp per bitmap word: the kept blocks' live positions
#include <float.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kScoreWarps = 8;
constexpr int kTopkThreads = 512;
constexpr int kMaxSelQueries = 8;
constexpr int kMaxSelFeatures = 1024;
constexpr int kMaxSelBlocks = 16384;

struct SelParams {
    const float *q_idx;      // [B][T][F]
    const uint16_t *pooled;  // [B][NB][F] bf16 bits
    const int32_t *n_live;   // [B]
    const int32_t *steps;    // [B][T] or nullptr
    float *scores;           // [B][T][NB]
    int32_t *kept;           // [B][T][K]
    int32_t *sel;            // concatenated positions
    int32_t *sel_offsets;    // [B+1]
    uint32_t *bitmap;        // [B][W]
    int32_t *word_pre;       // [B][W] positions before the word
    int32_t *seq_cells;      // [B]
    uint32_t *ticket;        // [1 + B]: sequences counted, then each sequence's finished queries
    uint32_t *status;
    int32_t n_seq, T, F, R, NB, K, W;
};

// Live positions of sequence b, clamped to the capacity (a bad value is
// reported by the scorer's first CTA of the sequence).
__device__ __forceinline__ int live_of(const SelParams &p, int b)
{
    const int v = __ldg(p.n_live + b);
    const long long cap = (long long)p.NB * p.R;
    return v < 0 ? 0 : (v > cap ? (int)cap : v);
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// ---------------------------------------------------------------- scores

constexpr int kMaxChunksPerLane = kMaxSelFeatures / 8 / 32; // 16-byte pieces of a key per lane

// CPL: 16-byte pieces of a key per lane (F / 256, rounded up); BPW: blocks
// per warp, all their keys loaded before any is used.  BPW * CPL stays at 4,
// so a warp has 2 KB of keys in flight and the grid (NB / (8 BPW) CTAs per
// sequence) fits the SMs in one wave at the sizes of a long context.
template <int CPL, int BPW>
__global__ void __launch_bounds__(kScoreWarps * 32, 1) qsa_block_scores_kernel(const SelParams p)
{
    extern __shared__ __align__(16) float s_q[]; // [T][F]
    const int b = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j0 = blockIdx.x * (BPW * kScoreWarps);
    const int live = live_of(p, b);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int v = __ldg(p.n_live + b);
        if ((v < 0 || (long long)v > (long long)p.NB * p.R) && p.status) atomicOr(p.status, QSA_STATUS_BAD_EXTENT);
        p.ticket[1 + b] = 0u;      // the top-k's per-sequence completion ticket
        if (b == 0) *p.ticket = 0; // and the sequences' ticket
    }
    // the top-k may launch now: it waits for this grid before it reads
    cudaTriggerProgrammaticLaunchCompletion();
    // empty bitmap words for the top-k to OR into: the CTA that holds a
    // word's first block clears it
    if (threadIdx.x == 0 && (j0 & 31) == 0) p.bitmap[(size_t)b * p.W + j0 / 32] = 0u;
    const float *q = p.q_idx + (size_t)b * p.T * p.F;
    for (int e = threadIdx.x; e < p.T * p.F; e += blockDim.x) s_q[e] = __ldg(q + e);
    __syncthreads();
    const int nchunk = p.F / 8; // 16-byte pieces of a pooled key
    int jb[BPW];
    bool live_blk[BPW];
    uint4 kw[BPW][CPL];
#pragma unroll
    for (int u = 0; u < BPW; ++u) {
        jb[u] = j0 + warp + kScoreWarps * u;
        live_blk[u] = jb[u] < p.NB && (long long)jb[u] * p.R < live;
        const uint16_t *key = p.pooled + ((size_t)b * p.NB + (live_blk[u] ? jb[u] : 0)) * p.F;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int ch = lane + 32 * c;
            kw[u][c] = make_uint4(0, 0, 0, 0);
            if (live_blk[u] && ch < nchunk) kw[u][c] = ldg_nc_v4(key + 8 * ch);
        }
    }
#pragma unroll
    for (int u = 0; u < BPW; ++u) {
        const int j = jb[u];
        if (j >= p.NB) continue;
        float acc[kMaxSelQueries];
#pragma unroll
        for (int t = 0; t < kMaxSelQueries; ++t) acc[t] = 0.f;
        if (live_blk[u]) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ch = lane + 32 * c;
                if (ch < nchunk) {
                    const uint4 w = kw[u][c];
                    const float k8[8] = {bf16_to_f32(w.x & 0xffffu), bf16_to_f32(w.x >> 16),
                                         bf16_to_f32(w.y & 0xffffu), bf16_to_f32(w.y >> 16),
                                         bf16_to_f32(w.z & 0xffffu), bf16_to_f32(w.z >> 16),
                                         bf16_to_f32(w.w & 0xffffu), bf16_to_f32(w.w >> 16)};
#pragma unroll
                    for (int t = 0; t < kMaxSelQueries; ++t) {
                        if (t < p.T) {
                            const float4 qa = *reinterpret_cast<const float4 *>(s_q + t * p.F + 8 * ch);
                            const float4 qb = *reinterpret_cast<const float4 *>(s_q + t * p.F + 8 * ch + 4);
                            float a = acc[t];
                            a = fmaf(qa.x, k8[0], a); a = fmaf(qa.y, k8[1], a);
                            a = fmaf(qa.z, k8[2], a); a = fmaf(qa.w, k8[3], a);
                            a = fmaf(qb.x, k8[4], a); a = fmaf(qb.y, k8[5], a);
                            a = fmaf(qb.z, k8[6], a); a = fmaf(qb.w, k8[7], a);
                            acc[t] = a;
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kMaxSelQueries; ++t)
                if (t < p.T)
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
        }
        if (lane < p.T) {
            float a = acc[0];
#pragma unroll
            for (int t = 1; t < kMaxSelQueries; ++t)
                if (lane == t) a = acc[t];
            const bool cand = live_blk[u] && (p.steps == nullptr || (long long)j * p.R <= (long long)__ldg(p.steps + (size_t)b * p.T + lane));
            p.scores[((size_t)b * p.T + lane) * p.NB + j] = cand ? a : -INFINITY;
        }
    }
}

// ---------------------------------------------------------------- top-k

// Order-preserving 32-bit key of a float (larger float, larger key); -inf
// has the smallest key of all non-NaN values.
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan over the CTA of one value per thread (fixed order).
__device__ __forceinline__ int block_exclusive_scan(int v, int *s_warp, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? s_warp[lane] : 0;
        int ws = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += y;
        }
        if (lane < nw) s_warp[lane] = ws - w; // exclusive
        if (lane == nw - 1) s_warp[32] = ws;
    }
    __syncthreads();
    const int r = s_warp[warp] + x - v;
    *total = s_warp[32];
    __syncthreads();
    return r;
}

// Positions of the kept blocks in bitmap word w of sequence b.
__device__ __forceinline__ int word_cells(const SelParams &p, uint32_t bits, int w, int live)
{
    if (!bits) return 0;
    int cells = __popc(bits) * p.R;
    // only the last live block can be partial
    const int last = (live + p.R - 1) / p.R - 1; // last live block (live > 0 when bits != 0)
    if (last >= 32 * w && last < 32 * w + 32 && (bits >> (last - 32 * w)) & 1u)
        cells -= (last + 1) * p.R - live;
    return cells;
}

__global__ void __launch_bounds__(kTopkThreads) qsa_topk_kernel(const SelParams p)
{
    extern __shared__ __align__(16) uint32_t s_key[]; // [NB]
    __shared__ int s_hist[256];
    __shared__ int s_warp[33];
    __shared__ uint32_t s_bits[kMaxSelBlocks / 32];
    __shared__ int s_pick[2];
    __shared__ bool s_last;
    const int bt = blockIdx.x, b = bt / p.T;
    const int n = p.NB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    // the expansion may launch now; it waits for this grid before it reads
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize(); // the scores, the cleared bitmap and tickets
    const float *sc = p.scores + (size_t)bt * n;
    // keys, and the number of candidates (finite scores)
    int fin = 0;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const float f = sc[j];
        s_key[j] = order_key(f);
        fin += f > -INFINITY;
    }
    for (int w = threadIdx.x; w < (n + 31) / 32; w += blockDim.x) s_bits[w] = 0u;
    int cnt;
    block_exclusive_scan(fin, s_warp, &cnt);
    const int kk = min(p.K, cnt);
    // the kk-th largest key: four passes over 8-bit digits, most significant
    // first, among the keys that share the digits found so far
    uint32_t prefix = 0u, mask = 0u;
    int need = kk; // keys still to take at or below the current prefix
    if (kk > 0) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = threadIdx.x; i < 256; i += blockDim.x) s_hist[i] = 0;
            __syncthreads();
            // a warp's lanes with the same digit add once, together
            for (int jw = 32 * warp; jw < n; jw += 32 * nwarps) {
                const int j = jw + lane;
                const uint32_t k = j < n ? s_key[j] : 0u;
                const bool in = j < n && (k & mask) == prefix;
                if (!__any_sync(0xffffffffu, in)) continue;
                // (the lanes out of the prefix form one group, which adds nothing)
                const uint32_t d = in ? (k >> shift) & 0xFFu : 0xFFFFFFFFu;
                const unsigned grp = __match_any_sync(0xffffffffu, d);
                if (in && lane == __ffs(grp) - 1) atomicAdd(&s_hist[d], __popc(grp));
            }
            __syncthreads();
            if (warp == 0) {
                // lane l holds digits 8l..8l+7: the digit at which the keys
                // counted from 255 down first reach `need`, and the count above it
                int c[8], lsum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    c[i] = s_hist[8 * lane + i];
                    lsum += c[i];
                }
                int suf = lsum; // keys with digits >= 8 * lane
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_down_sync(0xffffffffu, suf, o);
                    if (lane + o < 32) suf += v;
                }
                int above = suf - lsum;
                if (above < need && need <= suf) {
                    int d = 8 * lane;
#pragma unroll
                    for (int i = 7; i >= 0; --i) {
                        if (above + c[i] >= need) {
                            d = 8 * lane + i;
                            break;
                        }
                        above += c[i];
                    }
                    s_pick[0] = d;
                    s_pick[1] = above;
                }
            }
            __syncthreads();
            prefix |= (uint32_t)s_pick[0] << shift;
            mask |= 0xFFu << shift;
            need -= s_pick[1];
            __syncthreads();
        }
    }
    // kept: keys above the threshold, and the first `need` keys equal to it
    // in block order.  Thread i takes the contiguous blocks [i*per, (i+1)*per).
    const uint32_t thr = prefix;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int eq = 0;
    if (kk > 0)
        for (int j = lo; j < hi; ++j) eq += s_key[j] == thr;
    int eq_total;
    int eq_before = block_exclusive_scan(eq, s_warp, &eq_total);
    int mine = 0;
    if (kk > 0)
        for (int j = lo; j < hi; ++j) {
            const uint32_t k = s_key[j];
            const bool take = k > thr || (k == thr && eq_before++ < need);
            if (take) {
                ++mine;
                atomicOr(&s_bits[j >> 5], 1u << (j & 31));
            }
        }
    int total;
    int out = block_exclusive_scan(mine, s_warp, &total);
    int32_t *dst = p.kept + (size_t)bt * p.K;
    if (kk > 0)
        for (int j = lo; j < hi; ++j)
            if (s_bits[j >> 5] & (1u << (j & 31))) {
                if (out < p.K) dst[out] = j; // (exactly kk are kept; the guard only bounds the write)
                ++out;
            }
    for (int i = total + threadIdx.x; i < p.K; i += blockDim.x) dst[i] = -1;
    __syncthreads();
    for (int w = threadIdx.x; w < (n + 31) / 32; w += blockDim.x)
        if (s_bits[w]) atomicOr(p.bitmap + (size_t)b * p.W + w, s_bits[w]);
    // the last of the sequence's T CTAs counts its positions (per bitmap
    // word, a scan); the last sequence counted scans the sequences into
    // the CSR offsets
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.ticket + 1 + b, 1u) == (unsigned)p.T - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int live = live_of(p, b);
    int run = 0;
    for (int w0 = 0; w0 < p.W; w0 += blockDim.x) {
        const int w = w0 + threadIdx.x;
        const uint32_t bits = w < p.W ? *reinterpret_cast<volatile uint32_t *>(p.bitmap + (size_t)b * p.W + w) : 0u;
        const int c = w < p.W ? word_cells(p, bits, w, live) : 0;
        int tot;
        const int before = block_exclusive_scan(c, s_warp, &tot);
        if (w < p.W) p.word_pre[(size_t)b * p.W + w] = run + before;
        run += tot;
    }
    if (threadIdx.x == 0) p.seq_cells[b] = run;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.ticket, 1u) == (unsigned)p.n_seq - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    int base = 0;
    for (int b0 = 0; b0 < p.n_seq; b0 += blockDim.x) {
        const int i = b0 + threadIdx.x;
        const int c = i < p.n_seq ? *reinterpret_cast<volatile int32_t *>(p.seq_cells + i) : 0;
        int tot;
        const int before = block_exclusive_scan(c, s_warp, &tot);
        if (i < p.n_seq) p.sel_offsets[i] = base + before;
        base += tot;
    }
    if (threadIdx.x == 0) p.sel_offsets[p.n_seq] = base;
}

// ---------------------------------------------------------------- expand

__global__ void __launch_bounds__(256) qsa_select_expand_kernel(const SelParams p)
{
    const int b = blockIdx.y, lane = threadIdx.x & 31;
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5);
    cudaGridDependencySynchronize(); // the bitmap, the word prefixes and the offsets
    if (w >= p.W) return;
    uint32_t bits = p.bitmap[(size_t)b * p.W + w];
    if (!bits) return;
    const int live = live_of(p, b);
    int base = p.sel_offsets[b] + p.word_pre[(size_t)b * p.W + w];
    while (bits) {
        const int j = 32 * w + __ffs(bits) - 1;
        bits &= bits - 1;
        const int start = j * p.R;
        const int cells = min(p.R, live - start);
        for (int i = lane; i < cells; i += 32) p.sel[base + i] = start + i;
        base += cells;
    }
}

struct SelWorkspace {
    size_t off_bitmap, off_pre, off_cells, off_ticket, total;
};

SelWorkspace sel_carve(const qsa_select_shape *s, int n_seq)
{
    const size_t W = ((size_t)s->max_blocks + 31) / 32;
    SelWorkspace w{};
    w.off_bitmap = 0;
    w.off_pre = align_up(w.off_bitmap + (size_t)n_seq * W * 4, 256);
    w.off_cells = align_up(w.off_pre + (size_t)n_seq * W * 4, 256);
    w.off_ticket = align_up(w.off_cells + (size_t)n_seq * 4, 256);
    w.total = align_up(w.off_ticket + 4 * ((size_t)n_seq + 1), 256);
    return w;
}

qsa_status sel_check(const qsa_select_shape *s)
{
    if (!s) return QSA_ERR_INVALID_ARG;
    if (s->n_queries < 1 || s->idx_heads < 1 || s->idx_dim < 1 || s->block_cells < 1 || s->max_blocks < 1 ||
        s->top_k < 1)
        return QSA_ERR_INVALID_ARG;
    const long long F = (long long)s->idx_heads * s->idx_dim;
    if (s->n_queries > kMaxSelQueries || F > kMaxSelFeatures || F % 8 != 0 || s->max_blocks > kMaxSelBlocks ||
        s->top_k > s->max_blocks || (long long)s->max_blocks * s->block_cells > 0x7fffffffll)
        return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

} // namespace
} // namespace qsa

extern "C" {

qsa_status qsa_select_workspace_bytes(const qsa_select_shape *shape, int32_t n_seq, size_t *bytes)
{
    const qsa_status st = qsa::sel_check(shape);
    if (st != QSA_OK) return st;
    if (!bytes || n_seq < 1) return QSA_ERR_INVALID_ARG;
    *bytes = qsa::sel_carve(shape, n_seq).total;
    return QSA_OK;
}

qsa_status qsa_select_blocks(const qsa_select_shape *shape, int32_t n_seq, const float *q_idx,
                             const uint16_t *pooled, const int32_t *n_live, const int32_t *steps,
                             float *scores, int32_t *kept, int32_t *sel, int32_t *sel_offsets,
                             void *workspace, size_t workspace_bytes, uint32_t *status, void *stream)
{
    using namespace qsa;
    qsa_status st = sel_check(shape);
    if (st != QSA_OK) return st;
    if (n_seq < 1 || n_seq > 65535 || !q_idx || !pooled || !n_live || !scores || !kept || !sel ||
        !sel_offsets || !workspace)
        return QSA_ERR_INVALID_ARG;
    auto al = [](const void *ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; };
    if (!al(q_idx, 16) || !al(pooled, 16) || !al(n_live, 4) || (steps && !al(steps, 4)) || !al(scores, 4) ||
        !al(kept, 4) || !al(sel, 4) || !al(sel_offsets, 4) || !al(workspace, 256) || (status && !al(status, 4)))
        return QSA_ERR_INVALID_ARG;
    const SelWorkspace w = sel_carve(shape, n_seq);
    if (workspace_bytes < w.total) return QSA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    SelParams p{};
    p.q_idx = q_idx;
    p.pooled = pooled;
    p.n_live = n_live;
    p.steps = steps;
    p.scores = scores;
    p.kept = kept;
    p.sel = sel;
    p.sel_offsets = sel_offsets;
    p.bitmap = reinterpret_cast<uint32_t *>(ws + w.off_bitmap);
    p.word_pre = reinterpret_cast<int32_t *>(ws + w.off_pre);
    p.seq_cells = reinterpret_cast<int32_t *>(ws + w.off_cells);
    p.ticket = reinterpret_cast<uint32_t *>(ws + w.off_ticket);
    p.status = status;
    p.n_seq = n_seq;
    p.T = shape->n_queries;
    p.F = shape->idx_heads * shape->idx_dim;
    p.R = shape->block_cells;
    p.NB = shape->max_blocks;
    p.K = shape->top_k;
    p.W = (p.NB + 31) / 32;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const size_t q_smem = (size_t)p.T * p.F * sizeof(float);
    // the scorer waits for everything before it on the stream (it clears the
    // bitmap and tickets the previous call's kernels read)
    auto sgrid = [&](int bpw) {
        return dim3((unsigned)((p.NB + bpw * kScoreWarps - 1) / (bpw * kScoreWarps)), (unsigned)n_seq);
    };
    switch ((p.F / 8 + 31) / 32) {
    case 1: qsa_block_scores_kernel<1, 4><<<sgrid(4), kScoreWarps * 32, q_smem, cs>>>(p); break;
    case 2: qsa_block_scores_kernel<2, 2><<<sgrid(2), kScoreWarps * 32, q_smem, cs>>>(p); break;
    case 3: qsa_block_scores_kernel<3, 1><<<sgrid(1), kScoreWarps * 32, q_smem, cs>>>(p); break;
    default: qsa_block_scores_kernel<kMaxChunksPerLane, 1><<<sgrid(1), kScoreWarps * 32, q_smem, cs>>>(p); break;
    }
    if (cudaGetLastError() != cudaSuccess) return QSA_ERR_CUDA;
    const int key_smem = p.NB * 4;
    if (cudaFuncSetAttribute(qsa_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, key_smem) != cudaSuccess)
        return QSA_ERR_CUDA;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_seq * p.T));
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = (size_t)key_smem;
    cfg.stream = cs;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, qsa_topk_kernel, p) != cudaSuccess) return QSA_ERR_CUDA;
    cfg.gridDim = dim3((unsigned)((p.W + 7) / 8), (unsigned)n_seq);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, qsa_select_expand_kernel, p) != cudaSuccess) return QSA_ERR_CUDA;
    return QSA_OK;
}

} // extern "C"
