// qsa_merge.cu -- split-K merge of chunk partials (step a5).
//
// The pages' decode attention is "chunk kernel + merge" ("Strata PR #2220,
// attn_chunk_q8_v3_kernel", opening description and kernel table).  Chunk c
// of a row carries (m_c, l_c, o_c) with m in natural-log units; the merge is
//   M = max_{c: l_c > 0} m_c,  L = sum_c l_c e^{m_c - M},
//   out = sum_c o_c e^{m_c - M} / L   (zeros when no chunk holds a cell).
// A CTA of four warps covers four query rows with one warp each when a row
// has at most four chunks, or one row with all four warps otherwise (warp w
// takes chunks w, w+4, ...).  Lane k owns output dimensions 8k..8k+7.  Each
// warp forms its own (M_w, L_w, acc_w), four chunks at a time with all their
// loads in flight together and a running maximum; with four warps per row
// their results are then combined in shared memory.  Every sum runs in a
// fixed order, so the output is bit-identical from run to run.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kMergeWarps = 4;

template <int WPR> // warps per row: 1 or kMergeWarps
__global__ void __launch_bounds__(kMergeWarps * 32) qsa_merge_kernel(const Params p)
{
    __shared__ float s_acc[kMergeWarps][kHeadDim];
    __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
    const int lane = threadIdx.x & 31;
    const int w = WPR == 1 ? 0 : threadIdx.x >> 5; // this warp's first chunk
    const int r = WPR == 1 ? blockIdx.x * kMergeWarps + (threadIdx.x >> 5) : blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    // launched as a programmatic dependent of the chunk kernel: wait until
    // that grid has finished and its partials are visible
    cudaGridDependencySynchronize();
    if (r >= p.R) return;
    const size_t base = ((size_t)b * p.G + g) * p.n_chunks * p.R + r;
    const size_t stride = (size_t)p.R; // chunk stride of m and l
    // chunks are taken four at a time with every load of a group issued
    // together (the list length is only needed to mask the group, so its
    // read overlaps the first group's), combined with a running maximum
    int start, n;
    seq_range(p, b, &start, &n);
    float M = -INFINITY, Lpart = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c0 = w; c0 < p.n_chunks; c0 += 4 * WPR) {
        float mu[4], lu[4];
        float4 ou[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * WPR;
            mu[u] = -INFINITY;
            lu[u] = 0.f;
            if (c < p.n_chunks) {
                const size_t idx = base + (size_t)c * stride;
                mu[u] = p.part_m[idx];
                lu[u] = p.part_l[idx];
                const float4 *src = reinterpret_cast<const float4 *>(p.part_o + idx * kHeadDim + lane * 8);
                ou[u][0] = src[0];
                ou[u][1] = src[1];
            }
        }
        const int n_chunks = n > 0 ? (n + p.chunk_cells - 1) / p.chunk_cells : 0;
        bool ok[4];
        float gm = -INFINITY;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            ok[u] = c0 + u * WPR < n_chunks && lu[u] > 0.f;
            if (ok[u]) gm = fmaxf(gm, mu[u]);
        }
        if (gm > M) {
            const float f = M == -INFINITY ? 0.f : expf(M - gm);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] *= f;
            Lpart *= f;
            M = gm;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (!ok[u]) continue;
            const float wu = mu[u] == M ? 1.f : expf(mu[u] - M);
            Lpart = fmaf(lu[u], wu, Lpart);
            acc[0] = fmaf(ou[u][0].x, wu, acc[0]);
            acc[1] = fmaf(ou[u][0].y, wu, acc[1]);
            acc[2] = fmaf(ou[u][0].z, wu, acc[2]);
            acc[3] = fmaf(ou[u][0].w, wu, acc[3]);
            acc[4] = fmaf(ou[u][1].x, wu, acc[4]);
            acc[5] = fmaf(ou[u][1].y, wu, acc[5]);
            acc[6] = fmaf(ou[u][1].z, wu, acc[6]);
            acc[7] = fmaf(ou[u][1].w, wu, acc[7]);
        }
        if (c0 + 4 * WPR >= n_chunks) break;
    }
    const int t = r / p.H, j = r % p.H;
    float *orow = p.out + (((size_t)b * p.T + t) * p.G * p.H + (size_t)g * p.H + j) * kHeadDim;
    if (WPR == 1) {
        float4 *dst = reinterpret_cast<float4 *>(orow + lane * 8);
        const float L = Lpart;
        if (L > 0.f) {
            dst[0] = make_float4(acc[0] / L, acc[1] / L, acc[2] / L, acc[3] / L);
            dst[1] = make_float4(acc[4] / L, acc[5] / L, acc[6] / L, acc[7] / L);
        } else {
            dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    *reinterpret_cast<float4 *>(&s_acc[w][lane * 8]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4 *>(&s_acc[w][lane * 8 + 4]) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if (lane == 0) {
        s_m[w] = M;
        s_l[w] = Lpart;
    }
    __syncthreads();

    // combine the warps' results (fixed order); thread t owns dimensions 2t, 2t+1
    float Mt = -INFINITY;
#pragma unroll
    for (int x = 0; x < kMergeWarps; ++x)
        if (s_l[x] > 0.f) Mt = fmaxf(Mt, s_m[x]);
    float L = 0.f, o0 = 0.f, o1 = 0.f;
    if (Mt > -INFINITY) {
#pragma unroll
        for (int x = 0; x < kMergeWarps; ++x) {
            if (!(s_l[x] > 0.f)) continue;
            const float f = s_m[x] == Mt ? 1.f : expf(s_m[x] - Mt);
            L = fmaf(s_l[x], f, L);
            o0 = fmaf(s_acc[x][2 * threadIdx.x], f, o0);
            o1 = fmaf(s_acc[x][2 * threadIdx.x + 1], f, o1);
        }
    }
    float2 *dst = reinterpret_cast<float2 *>(orow + 2 * threadIdx.x);
    *dst = L > 0.f ? make_float2(o0 / L, o1 / L) : make_float2(0.f, 0.f);
}

} // namespace

cudaError_t launch_merge(const Params &p, cudaStream_t stream)
{
    // one warp per row when rows have few chunks, four otherwise
    const bool wide = p.n_chunks > kMergeWarps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(wide ? p.R : (p.R + kMergeWarps - 1) / kMergeWarps), (unsigned)p.G, (unsigned)p.n_seq);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return wide ? cudaLaunchKernelEx(&cfg, qsa_merge_kernel<kMergeWarps>, p)
                : cudaLaunchKernelEx(&cfg, qsa_merge_kernel<1>, p);
}

} // namespace qsa
