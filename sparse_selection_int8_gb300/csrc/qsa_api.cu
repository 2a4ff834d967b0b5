// qsa_api.cu -- the C ABI declared in include/qsa.h: argument checks,
// workspace carve-up, kernel choice and launches.  Nothing here allocates,
// synchronises or keeps state between calls.
#include <math.h>
#include <string.h>

#include <atomic>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kMaxRowsPerKv = 64 * 65536; // q_per_kv <= 64, n_queries <= 65536
constexpr size_t kWorkspaceAlign = 256;
constexpr long long kDefaultWaitCycles = 1ll << 32; // about two seconds of SM clock

// Bound of the kernels' device-side waits (qsa_set_wait_limit; 0 = default).
std::atomic<long long> g_wait_cycles{0};

bool aligned(const void *ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

qsa_status check_shape(const qsa_shape *s)
{
    if (!s) return QSA_ERR_INVALID_ARG;
    if (s->n_kv_heads < 1 || s->q_per_kv < 1 || s->n_queries < 1 || s->pool_cells < 1 ||
        s->page_table_len < 1 || s->chunk_cells < 1)
        return QSA_ERR_INVALID_ARG;
    if (!isfinite(s->softmax_scale)) return QSA_ERR_INVALID_ARG;
    if (s->q_dtype != QSA_F32 && s->q_dtype != QSA_BF16) return QSA_ERR_INVALID_ARG;
    if (s->algo != QSA_ALGO_AUTO && s->algo != QSA_ALGO_SIMT && s->algo != QSA_ALGO_TCGEN05)
        return QSA_ERR_INVALID_ARG;
    if (s->page_cells < 0) return QSA_ERR_INVALID_ARG;
    const int P = s->page_cells > 0 ? s->page_cells : 1;
    if (s->pool_cells % P != 0 || (long long)s->page_table_len * P > 0x7fffffffll)
        return QSA_ERR_INVALID_ARG;
    if (s->head_dim != kHeadDim) return QSA_ERR_UNSUPPORTED;
    if (s->q_per_kv > 64 || s->n_queries > 65536 || s->n_kv_heads > 65535)
        return QSA_ERR_UNSUPPORTED;
    if ((long long)s->q_per_kv * s->n_queries > kMaxRowsPerKv) return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

enum Path { kPathSimt = 0, kPathDecodeTc = 1, kPathPromptTc = 2, kPathNone = -1 };

// Kernel family by shape: the cells-on-M tensor-core kernel for decode
// windows (at most 80 query rows per KV head), the rows-on-M tensor-core
// kernel for prompt-shaped calls (chunks of at least one 128-cell tile), the
// CUDA-core kernel otherwise or when asked for.
Path select_path(const qsa_shape *s)
{
    const long long R = (long long)s->q_per_kv * s->n_queries;
    if (s->algo == QSA_ALGO_SIMT) return kPathSimt;
    if (R <= kDecodeTcMaxRows) return kPathDecodeTc;
    if (s->chunk_cells >= 128) return kPathPromptTc;
    return s->algo == QSA_ALGO_TCGEN05 ? kPathNone : kPathSimt;
}

Workspace carve(const qsa_shape *s, int n_seq, int max_selected)
{
    Workspace w{};
    const size_t R = (size_t)s->q_per_kv * s->n_queries;
    const size_t n_chunks = max_selected > 0 ? ((size_t)max_selected + s->chunk_cells - 1) / s->chunk_cells : 0;
    const size_t rows = (size_t)n_seq * s->n_kv_heads * n_chunks * R;
    w.off_m = 0;
    w.off_l = align_up(w.off_m + rows * sizeof(float), kWorkspaceAlign);
    w.off_o = align_up(w.off_l + rows * sizeof(float), kWorkspaceAlign);
    w.off_extra = align_up(w.off_o + rows * kHeadDim * sizeof(float), 1024);
    w.total = w.off_extra;
    if (select_path(s) == kPathDecodeTc && n_chunks > 0) {
        w.off_runs = w.off_extra + align_up(chunk_tc_query_image_bytes(n_seq, s->n_kv_heads, (int)R), 1024);
        w.total = w.off_runs + align_up((size_t)n_seq * s->n_kv_heads * sizeof(int32_t), kWorkspaceAlign);
    }
    if (select_path(s) == kPathPromptTc && n_chunks > 0) {
        size_t kb, qb, cb;
        prompt_image_bytes(n_seq, s->n_kv_heads, (int)R, s->chunk_cells, (int)n_chunks, &kb, &qb, &cb);
        w.total = w.off_extra + 2 * align_up(kb, 1024) + align_up(qb, 1024) + 3 * align_up(cb, 1024);
    }
    return w;
}

PromptImages prompt_images(const qsa_shape *s, int n_seq, int max_selected, char *ws, const Workspace &w)
{
    PromptImages im{};
    const int R = s->q_per_kv * s->n_queries;
    const int n_chunks = max_selected > 0 ? (max_selected + s->chunk_cells - 1) / s->chunk_cells : 0;
    size_t kb, qb, cb;
    prompt_image_bytes(n_seq, s->n_kv_heads, R, s->chunk_cells, n_chunks, &kb, &qb, &cb);
    size_t off = w.off_extra;
    im.k = ws + off;
    off += align_up(kb, 1024);
    im.v = ws + off;
    off += align_up(kb, 1024);
    im.q = ws + off;
    off += align_up(qb, 1024);
    im.ksc = reinterpret_cast<float *>(ws + off);
    off += align_up(cb, 1024);
    im.bias = reinterpret_cast<float *>(ws + off);
    off += align_up(cb, 1024);
    im.pos = reinterpret_cast<int32_t *>(ws + off);
    im.tiles_per_chunk = (s->chunk_cells + 127) / 128;
    im.row_tiles = (R + 127) / 128;
    return im;
}

qsa_status run(const qsa_shape *s, int n_seq, const void *q, const int8_t *k_pool,
               const int8_t *v_pool, const float *k_scale, const float *v_scale,
               const int32_t *page_table, const int32_t *sel, const int32_t *sel_offsets,
               int n_sel_single, int max_selected, float *out, void *workspace,
               size_t workspace_bytes, uint32_t *status, void *stream,
               const int32_t *q_limit = nullptr)
{
    qsa_status st = check_shape(s);
    if (st != QSA_OK) return st;
    if (n_seq < 1 || n_seq > 65535 || max_selected < 0) return QSA_ERR_INVALID_ARG;
    if (!q || !k_pool || !v_pool || !k_scale || !v_scale || !page_table || !out)
        return QSA_ERR_INVALID_ARG;
    if (max_selected > 0 && !sel) return QSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
        !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(page_table, 4) ||
        (sel && !aligned(sel, 4)) || (status && !aligned(status, 4)) ||
        (q_limit && !aligned(q_limit, 4)))
        return QSA_ERR_INVALID_ARG;
    if ((const void *)out == q || (const void *)out == (const void *)k_pool ||
        (const void *)out == (const void *)v_pool)
        return QSA_ERR_INVALID_ARG;
    const Workspace w = carve(s, n_seq, max_selected);
    if (w.total > 0 && (!workspace || !aligned(workspace, kWorkspaceAlign)))
        return QSA_ERR_INVALID_ARG;
    if (workspace_bytes < w.total) return QSA_ERR_WORKSPACE;

    Params p{};
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.page_table = page_table;
    p.sel = sel;
    p.sel_offsets = sel_offsets;
    p.q_limit = q_limit;
    p.out = out;
    char *ws = static_cast<char *>(workspace);
    p.part_m = reinterpret_cast<float *>(ws + w.off_m);
    p.part_l = reinterpret_cast<float *>(ws + w.off_l);
    p.part_o = reinterpret_cast<float *>(ws + w.off_o);
    p.status = status;
    p.q_img = ws + w.off_extra;
    p.part_runs = w.off_runs > 0 ? reinterpret_cast<int32_t *>(ws + w.off_runs) : nullptr;
    p.n_sel_single = n_sel_single;
    p.n_seq = n_seq;
    p.G = s->n_kv_heads;
    p.H = s->q_per_kv;
    p.T = s->n_queries;
    p.R = s->q_per_kv * s->n_queries;
    p.pool_cells = s->pool_cells;
    p.page_table_len = s->page_table_len;
    p.page_cells = s->page_cells > 0 ? s->page_cells : 1;
    p.pool_pages = s->pool_cells / p.page_cells;
    p.chunk_cells = s->chunk_cells;
    p.max_selected = max_selected;
    p.n_chunks = max_selected > 0 ? (max_selected + s->chunk_cells - 1) / s->chunk_cells : 0;
    p.q_bf16 = s->q_dtype == QSA_BF16;
    p.scale_log2 = s->softmax_scale * kLog2e;
    const long long wl = g_wait_cycles.load(std::memory_order_relaxed);
    p.wait_cycles = wl > 0 ? wl : kDefaultWaitCycles;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const Path path = select_path(s);
    if (path == kPathNone) return QSA_ERR_UNSUPPORTED;
    cudaError_t e;
    if (path == kPathDecodeTc)
        e = launch_chunk_tc(p, cs);
    else if (path == kPathPromptTc)
        e = launch_prompt_tc(p, prompt_images(s, n_seq, max_selected, ws, w), cs);
    else
        e = launch_chunk_simt(p, cs);
    if (e != cudaSuccess) return QSA_ERR_CUDA;
    e = launch_merge(p, cs);
    if (e != cudaSuccess) return QSA_ERR_CUDA;
    return QSA_OK;
}

} // namespace
} // namespace qsa

extern "C" {

qsa_status qsa_workspace_bytes(const qsa_shape *shape, int32_t n_seq, int32_t max_selected,
                               size_t *bytes)
{
    qsa_status st = qsa::check_shape(shape);
    if (st != QSA_OK) return st;
    if (!bytes || n_seq < 1 || max_selected < 0) return QSA_ERR_INVALID_ARG;
    *bytes = qsa::carve(shape, n_seq, max_selected).total;
    return QSA_OK;
}

qsa_status qsa_decode_attn_step(const qsa_shape *shape, const void *q, const int8_t *k_pool,
                                const int8_t *v_pool, const float *k_scale,
                                const float *v_scale, const int32_t *page_table,
                                const int32_t *sel, int32_t n_sel, float *out, void *workspace,
                                size_t workspace_bytes, uint32_t *status, void *stream)
{
    if (n_sel < 0) return QSA_ERR_INVALID_ARG;
    return qsa::run(shape, 1, q, k_pool, v_pool, k_scale, v_scale, page_table, sel, nullptr,
                    n_sel, n_sel, out, workspace, workspace_bytes, status, stream);
}

qsa_status qsa_decode_attn_batch(const qsa_shape *shape, int32_t n_seq, const void *q,
                                 const int8_t *k_pool, const int8_t *v_pool,
                                 const float *k_scale, const float *v_scale,
                                 const int32_t *page_table, const int32_t *sel,
                                 const int32_t *sel_offsets, int32_t max_selected, float *out,
                                 void *workspace, size_t workspace_bytes, uint32_t *status,
                                 void *stream)
{
    if (!sel_offsets || !qsa::aligned(sel_offsets, 4)) return QSA_ERR_INVALID_ARG;
    return qsa::run(shape, n_seq, q, k_pool, v_pool, k_scale, v_scale, page_table, sel,
                    sel_offsets, 0, max_selected, out, workspace, workspace_bytes, status,
                    stream);
}

qsa_status qsa_decode_attn_batch_limited(const qsa_shape *shape, int32_t n_seq, const void *q,
                                         const int8_t *k_pool, const int8_t *v_pool,
                                         const float *k_scale, const float *v_scale,
                                         const int32_t *page_table, const int32_t *sel,
                                         const int32_t *sel_offsets, int32_t max_selected,
                                         const int32_t *q_limit, float *out, void *workspace,
                                         size_t workspace_bytes, uint32_t *status, void *stream)
{
    if (!sel_offsets || !qsa::aligned(sel_offsets, 4) || !q_limit) return QSA_ERR_INVALID_ARG;
    return qsa::run(shape, n_seq, q, k_pool, v_pool, k_scale, v_scale, page_table, sel,
                    sel_offsets, 0, max_selected, out, workspace, workspace_bytes, status,
                    stream, q_limit);
}

qsa_status qsa_partials_view(const qsa_shape *shape, int32_t n_seq, int32_t max_selected,
                             const void *workspace, const float **m, const float **l,
                             const float **o, int32_t *n_chunks)
{
    qsa_status st = qsa::check_shape(shape);
    if (st != QSA_OK) return st;
    if (n_seq < 1 || max_selected < 0 || !workspace) return QSA_ERR_INVALID_ARG;
    const qsa::Workspace w = qsa::carve(shape, n_seq, max_selected);
    const char *ws = static_cast<const char *>(workspace);
    if (m) *m = reinterpret_cast<const float *>(ws + w.off_m);
    if (l) *l = reinterpret_cast<const float *>(ws + w.off_l);
    if (o) *o = reinterpret_cast<const float *>(ws + w.off_o);
    if (n_chunks)
        *n_chunks = max_selected > 0 ? (max_selected + shape->chunk_cells - 1) / shape->chunk_cells : 0;
    return QSA_OK;
}

void qsa_set_wait_limit(int64_t cycles)
{
    qsa::g_wait_cycles.store(cycles > 0 ? (long long)cycles : 0, std::memory_order_relaxed);
}

const char *qsa_status_string(int32_t status)
{
    switch (status) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument";
    case QSA_ERR_UNSUPPORTED: return "unsupported shape";
    case QSA_ERR_WORKSPACE: return "workspace too small";
    case QSA_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
    }
}

} // extern "C"
