// qsa_merge.cu -- split-K merge of chunk partials (step a5).
//
// The pages' decode attention is "chunk kernel + merge" ("Strata PR #2220,
// attn_chunk_q8_v3_kernel", opening description and kernel table).  Chunk c
// of a row carries (m_c, l_c, o_c) with m in natural-log units; the merge is
//   M = max_{c: l_c > 0} m_c,  L = sum_c l_c e^{m_c - M},
//   out = sum_c o_c e^{m_c - M} / L   (zeros when no chunk holds a cell).
// One CTA per (row, KV head, sequence); thread d owns output dimension d and
// walks the chunks in ascending order, so the result is deterministic.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

__global__ void __launch_bounds__(kHeadDim) qsa_merge_kernel(const Params p)
{
    const int r = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int d = threadIdx.x;
    int start, n;
    seq_range(p, b, &start, &n);
    const int n_chunks = n > 0 ? (n + p.chunk_cells - 1) / p.chunk_cells : 0;
    const size_t base = ((size_t)b * p.G + g) * p.n_chunks * p.R + r;

    float M = -INFINITY;
    for (int c = 0; c < n_chunks; ++c) {
        const size_t idx = base + (size_t)c * p.R;
        if (p.part_l[idx] > 0.f) M = fmaxf(M, p.part_m[idx]);
    }
    float acc = 0.f, L = 0.f;
    if (M > -INFINITY) {
        for (int c = 0; c < n_chunks; ++c) {
            const size_t idx = base + (size_t)c * p.R;
            const float lc = p.part_l[idx];
            if (!(lc > 0.f)) continue;
            const float f = expf(p.part_m[idx] - M);
            L = fmaf(lc, f, L);
            acc = fmaf(p.part_o[idx * kHeadDim + d], f, acc);
        }
    }
    const int t = r / p.H, j = r % p.H;
    const size_t out_idx = (((size_t)b * p.T + t) * p.G * p.H + (size_t)g * p.H + j) * kHeadDim + d;
    p.out[out_idx] = L > 0.f ? acc / L : 0.f;
}

} // namespace

cudaError_t launch_merge(const Params &p, cudaStream_t stream)
{
    dim3 grid((unsigned)p.R, (unsigned)p.G, (unsigned)p.n_seq);
    qsa_merge_kernel<<<grid, kHeadDim, 0, stream>>>(p);
    return cudaGetLastError();
}

} // namespace qsa
