// qsa_merge.cu -- split-K merge of chunk partials (step a5).
//
// The pages' decode attention is "chunk kernel + merge" ("Strata PR #2220,
// attn_chunk_q8_v3_kernel", opening description and kernel table).  Chunk c
// of a row carries (m_c, l_c, o_c) with m in natural-log units; the merge is
//   M = max_{c: l_c > 0} m_c,  L = sum_c l_c e^{m_c - M},
//   out = sum_c o_c e^{m_c - M} / L   (zeros when no chunk holds a cell).
// One warp per query row: lane k owns output dimensions 8k..8k+7.  The
// lanes read the chunks' (m, l) pairs 32 at a time, form the weights
// e^{m_c - M} once, and broadcast them by shuffle while every lane sums its
// eight dimensions over the chunks with independent 16-byte loads.  All sums
// run in a fixed order (ascending chunks; a fixed shuffle tree for L), so the
// result is deterministic.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) qsa_merge_kernel(const Params p)
{
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    // launched as a programmatic dependent of the chunk kernel: wait until
    // that grid has finished and its partials are visible
    cudaGridDependencySynchronize();
    if (r >= p.R) return;
    int start, n;
    seq_range(p, b, &start, &n);
    const int n_chunks = n > 0 ? (n + p.chunk_cells - 1) / p.chunk_cells : 0;
    const size_t base = ((size_t)b * p.G + g) * p.n_chunks * p.R + r;
    const size_t stride = (size_t)p.R; // chunk stride of m and l

    float M = -INFINITY;
    for (int c = lane; c < n_chunks; c += 32) {
        const size_t idx = base + (size_t)c * stride;
        if (p.part_l[idx] > 0.f) M = fmaxf(M, p.part_m[idx]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float Lpart = 0.f;
    if (M > -INFINITY) {
        for (int c0 = 0; c0 < n_chunks; c0 += 32) {
            const int cnt = min(32, n_chunks - c0);
            float wgt = 0.f;
            if (lane < cnt) {
                const size_t idx = base + (size_t)(c0 + lane) * stride;
                const float lc = p.part_l[idx];
                if (lc > 0.f) {
                    wgt = expf(p.part_m[idx] - M);
                    Lpart = fmaf(lc, wgt, Lpart);
                }
            }
            const float *o = p.part_o + (base + (size_t)c0 * stride) * kHeadDim + lane * 8;
            const size_t ostride = stride * kHeadDim;
            int c = 0;
            for (; c + 4 <= cnt; c += 4) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 *src = reinterpret_cast<const float4 *>(o + (size_t)(c + u) * ostride);
                    v[2 * u] = src[0];
                    v[2 * u + 1] = src[1];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float wu = __shfl_sync(0xffffffffu, wgt, c + u);
                    acc[0] = fmaf(v[2 * u].x, wu, acc[0]);
                    acc[1] = fmaf(v[2 * u].y, wu, acc[1]);
                    acc[2] = fmaf(v[2 * u].z, wu, acc[2]);
                    acc[3] = fmaf(v[2 * u].w, wu, acc[3]);
                    acc[4] = fmaf(v[2 * u + 1].x, wu, acc[4]);
                    acc[5] = fmaf(v[2 * u + 1].y, wu, acc[5]);
                    acc[6] = fmaf(v[2 * u + 1].z, wu, acc[6]);
                    acc[7] = fmaf(v[2 * u + 1].w, wu, acc[7]);
                }
            }
            for (; c < cnt; ++c) {
                const float wu = __shfl_sync(0xffffffffu, wgt, c);
                const float4 *src = reinterpret_cast<const float4 *>(o + (size_t)c * ostride);
                const float4 a = src[0], b4 = src[1];
                acc[0] = fmaf(a.x, wu, acc[0]);
                acc[1] = fmaf(a.y, wu, acc[1]);
                acc[2] = fmaf(a.z, wu, acc[2]);
                acc[3] = fmaf(a.w, wu, acc[3]);
                acc[4] = fmaf(b4.x, wu, acc[4]);
                acc[5] = fmaf(b4.y, wu, acc[5]);
                acc[6] = fmaf(b4.z, wu, acc[6]);
                acc[7] = fmaf(b4.w, wu, acc[7]);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lpart += __shfl_xor_sync(0xffffffffu, Lpart, o);
    const float L = Lpart;
    const int t = r / p.H, j = r % p.H;
    float4 *dst = reinterpret_cast<float4 *>(
        p.out + (((size_t)b * p.T + t) * p.G * p.H + (size_t)g * p.H + j) * kHeadDim + lane * 8);
    if (L > 0.f) {
        dst[0] = make_float4(acc[0] / L, acc[1] / L, acc[2] / L, acc[3] / L);
        dst[1] = make_float4(acc[4] / L, acc[5] / L, acc[6] / L, acc[7] / L);
    } else {
        dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

} // namespace

cudaError_t launch_merge(const Params &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.R + kWarpsPerBlock - 1) / kWarpsPerBlock), (unsigned)p.G, (unsigned)p.n_seq);
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
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
