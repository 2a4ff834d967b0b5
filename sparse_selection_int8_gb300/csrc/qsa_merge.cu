// qsa_merge.cu -- split-K merge of chunk partials (step a5).
//
// The pages' decode attention is "chunk kernel + merge" ("Strata PR #2220,
// attn_chunk_q8_v3_kernel", opening description and kernel table).  Chunk c
// of a row carries (m_c, l_c, o_c) with m in natural-log units; the merge is
//   M = max_{c: l_c > 0} m_c,  L = sum_c l_c e^{m_c - M},
//   out = sum_c o_c e^{m_c - M} / L   (zeros when no chunk holds a cell).
// One CTA per (row, KV head, sequence).  The chunks' (m, l) pairs are read
// in parallel, 256 chunks at a time, into shared memory; the weights
// e^{m_c - M} are formed once per chunk; thread d then sums o_c[d] times its
// weight with independent loads.  Every sum runs in ascending chunk order,
// so the result is deterministic.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kBlock = kHeadDim; // one thread per output dimension

__global__ void __launch_bounds__(kBlock) qsa_merge_kernel(const Params p)
{
    __shared__ float s_w[kBlock];   // weights e^{m_c - M} (0 for empty chunks)
    __shared__ float s_lw[kBlock];  // l_c * weight
    __shared__ float s_red[kBlock / 32];
    const int r = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int d = threadIdx.x;
    // launched as a programmatic dependent of the chunk kernel: wait until
    // that grid has finished and its partials are visible
    cudaGridDependencySynchronize();
    int start, n;
    seq_range(p, b, &start, &n);
    const int n_chunks = n > 0 ? (n + p.chunk_cells - 1) / p.chunk_cells : 0;
    const size_t base = ((size_t)b * p.G + g) * p.n_chunks * p.R + r;

    // M: every thread takes chunks d, d+256, ...; then a block max (exact)
    float M = -INFINITY;
    for (int c = d; c < n_chunks; c += kBlock) {
        const size_t idx = base + (size_t)c * p.R;
        if (p.part_l[idx] > 0.f) M = fmaxf(M, p.part_m[idx]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((d & 31) == 0) s_red[d >> 5] = M;
    __syncthreads();
    M = s_red[0];
#pragma unroll
    for (int i = 1; i < kBlock / 32; ++i) M = fmaxf(M, s_red[i]);

    float acc = 0.f, L = 0.f;
    if (M > -INFINITY) {
        for (int c0 = 0; c0 < n_chunks; c0 += kBlock) {
            const int cnt = min(kBlock, n_chunks - c0);
            __syncthreads(); // the previous block's weights are consumed
            if (d < cnt) {
                const size_t idx = base + (size_t)(c0 + d) * p.R;
                const float lc = p.part_l[idx];
                const float wgt = lc > 0.f ? expf(p.part_m[idx] - M) : 0.f;
                s_w[d] = wgt;
                s_lw[d] = lc > 0.f ? lc * wgt : 0.f;
            }
            __syncthreads();
            const float *o = p.part_o + (base + (size_t)c0 * p.R) * kHeadDim + d;
            const size_t stride = (size_t)p.R * kHeadDim;
            int c = 0;
            for (; c + 4 <= cnt; c += 4) {
                const float o0 = o[(size_t)c * stride], o1 = o[(size_t)(c + 1) * stride];
                const float o2 = o[(size_t)(c + 2) * stride], o3 = o[(size_t)(c + 3) * stride];
                acc = fmaf(o0, s_w[c], acc);
                acc = fmaf(o1, s_w[c + 1], acc);
                acc = fmaf(o2, s_w[c + 2], acc);
                acc = fmaf(o3, s_w[c + 3], acc);
            }
            for (; c < cnt; ++c) acc = fmaf(o[(size_t)c * stride], s_w[c], acc);
            for (int cc = 0; cc < cnt; ++cc) L += s_lw[cc];
        }
    }
    const int t = r / p.H, j = r % p.H;
    const size_t out_idx = (((size_t)b * p.T + t) * p.G * p.H + (size_t)g * p.H + j) * kHeadDim + d;
    p.out[out_idx] = L > 0.f ? acc / L : 0.f;
}

} // namespace

cudaError_t launch_merge(const Params &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.R, (unsigned)p.G, (unsigned)p.n_seq);
    cfg.blockDim = dim3(kBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qsa_merge_kernel, p);
}

} // namespace qsa
