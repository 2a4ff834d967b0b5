// qsa_internal.cuh -- shared definitions of the QSA decode-attention kernels.
//
// Path of one call (the pages' "chunk kernel + merge", "Strata PR #2220,
// attn_chunk_q8_v3_kernel", opening description):
//   a1  selected list entry -> page-table slot (-1 masks the cell)
//   a2  INT8 K/V row gather + dequantise with the per-cell scales
//   a3  scores of every query row against every cell of the chunk
//   a4  chunk online softmax and P.V -> partials (m, l, o)
//   a5  split-K merge of the partials by log-sum-exp rescaling -> output
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qsa.h"

namespace qsa {

constexpr int kHeadDim = 256;
// Query rows (T x H of one KV head) the cells-on-M decode kernel takes; wider
// windows go to the rows-on-M kernel.
constexpr int kDecodeTcMaxRows = 80;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Everything a kernel needs about one call; passed by value.
struct Params {
    const void *q;             // [n_seq][T][G*H][D] f32 or bf16
    const int8_t *k_pool;      // [n_seq][G][pool][D]
    const int8_t *v_pool;
    const float *k_scale;      // [n_seq][G][pool]
    const float *v_scale;
    const int32_t *page_table; // [n_seq][N_log]
    const int32_t *sel;        // concatenated lists
    const int32_t *sel_offsets; // [n_seq+1] or nullptr (single sequence)
    const int32_t *q_limit;    // [n_seq][T] causal limits or nullptr: query t sees positions < limit
    float *out;                // [n_seq][T][G*H][D]
    float *part_m;             // [n_seq][G][n_chunks][R]
    float *part_l;
    float *part_o;             // [n_seq][G][n_chunks][R][D]
    int32_t *part_runs;        // decode tensor-core path: [n_seq][G] partial slots written
    int32_t runs;              // 1: slot k of a pair holds its k-th run of chunks (part_runs
                               // slots), 0: slot c holds chunk c
    int32_t merge_slots;       // slots per row the merge expects (its CTA shape; 0: n_chunks)
    uint32_t *status;          // optional
    void *q_img;               // decode tensor-core path: [n_seq][G] f16 query tiles (workspace)
    int32_t q_inline;          // decode tensor-core path, one (sequence, KV head): the chunk
                               // kernel converts the queries itself (no staging kernel)
    int32_t row_blocks;        // decode tensor-core path: the rows are split into this many
    int32_t rb_rows;           // blocks of rb_rows rows, each on its own CTAs (0 or 1: no split)
    int32_t n_sel_single;      // list length when sel_offsets == nullptr
    int32_t n_seq, G, H, T, R; // R = T*H rows per KV head
    int32_t pool_cells, page_table_len, chunk_cells, n_chunks, max_selected;
    int32_t page_cells;        // P >= 1: cells per page (positions: page_table_len * P)
    int32_t pool_pages;        // pool_cells / P: valid page entries are 0 .. pool_pages - 1
    int32_t q_bf16;
    float scale_log2;          // softmax_scale * log2(e)
    long long wait_cycles;     // bound of a device-side wait, SM clock cycles
};

// Tensor-core-ready operand images of the prompt-shaped path (workspace).
struct PromptImages {
    void *k;     // [n_seq][G][n_chunks][tiles_per_chunk] 64 KB tiles: K codes (bf16|f16)
    void *v;     // same tiles: f16(V code * v_scale)
    void *q;     // [n_seq][G][row_tiles] 64 KB tiles: queries (bf16|f16)
    float *ksc;  // [..][tiles_per_chunk][128]: k_scale * softmax_scale * log2(e), 0 if masked
    float *bias; // same: 0, or -inf for a masked cell
    int32_t *pos; // same: the cell's logical position (for causal limits)
    int tiles_per_chunk;
    int row_tiles;
};

// Workspace carve-up shared by the host code of every path.
struct Workspace {
    size_t off_m, off_l, off_o, off_extra, off_runs, total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__device__ __forceinline__ void raise_status(const Params &p, uint32_t bits)
{
    if (p.status) atomicOr(p.status, bits);
}

// List range of sequence b: [*start, *start + *n).  Bad offsets are clamped
// and reported instead of trusted.
__device__ __forceinline__ void seq_range(const Params &p, int b, int *start, int *n)
{
    if (p.sel_offsets == nullptr) {
        *start = 0;
        *n = p.n_sel_single;
        return;
    }
    int o0 = __ldg(p.sel_offsets + b);
    int o1 = __ldg(p.sel_offsets + b + 1);
    int len = o1 - o0;
    if (o0 < 0 || len < 0) {
        raise_status(p, QSA_STATUS_BAD_OFFSETS);
        *start = 0;
        *n = 0;
        return;
    }
    if (len > p.max_selected) {
        raise_status(p, QSA_STATUS_BAD_OFFSETS);
        len = p.max_selected;
    }
    *start = o0;
    *n = len;
}

// Step a1: logical position -> pool slot of sequence b; -1 when masked or
// out of range (out-of-range entries also raise a status bit).  Position pos
// lies on page pos / P at offset pos % P; the page entry (a page of the pool)
// places it at slot entry * P + offset.
__device__ __forceinline__ int resolve_slot(const Params &p, int b, int pos)
{
    const int P = p.page_cells;
    if (pos < 0 || (long long)pos >= (long long)p.page_table_len * P) {
        raise_status(p, QSA_STATUS_BAD_POSITION);
        return -1;
    }
    const int page = P == 1 ? pos : pos / P;
    const int e = __ldg(p.page_table + (size_t)b * p.page_table_len + page);
    if (e == -1) return -1;
    if (e < 0 || e >= p.pool_pages) {
        raise_status(p, QSA_STATUS_BAD_SLOT);
        return -1;
    }
    return P == 1 ? e : e * P + (pos - page * P);
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *ptr)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16)
{
    return __uint_as_float(bits16 << 16);
}

// Host-side launchers (defined in the kernel translation units).
cudaError_t launch_chunk_simt(const Params &p, cudaStream_t stream);
size_t chunk_tc_query_image_bytes(int n_seq, int G, int R);
cudaError_t launch_chunk_tc(Params &p, cudaStream_t stream); // sets p.runs, p.merge_slots
size_t prompt_image_bytes(int n_seq, int G, int R, int chunk_cells, int n_chunks, size_t *k_bytes,
                          size_t *q_bytes, size_t *cell_bytes);
cudaError_t launch_prompt_tc(const Params &p, const PromptImages &im, cudaStream_t stream);
cudaError_t launch_merge(const Params &p, cudaStream_t stream);

} // namespace qsa
