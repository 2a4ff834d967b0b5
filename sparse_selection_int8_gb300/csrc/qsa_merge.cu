// qsa_merge.cu -- split-K merge of chunk partials (step a5).
//
// The pages' decode attention is "chunk kernel + merge" ("Strata PR #2220,
// attn_chunk_q8_v3_kernel", opening description and kernel table).  Chunk c
// of a row carries (m_c, l_c, o_c) with m in natural-log units; the merge is
//   M = max_{c: l_c > 0} m_c,  L = sum_c l_c e^{m_c - M},
//   out = sum_c o_c e^{m_c - M} / L   (zeros when no chunk holds a cell).
// The tensor-core decode kernel may combine a run of consecutive chunks of a
// (sequence, KV head) into one partial (same m, l, o over the run's cells);
// then slots 0 .. part_runs[b][g] - 1 of the pair hold its runs, and the
// merge is the same over those slots.
// A CTA of four warps covers four query rows with one warp each when a row
// has at most four slots; otherwise a CTA of 2, 4 or 8 warps takes one row
// (warp w takes chunks w, w + WPR, ...), so one round of loads covers up to
// 4 * WPR chunks.  Lane k owns output dimensions 8k..8k+7.
// Each warp forms its own (M_w, L_w, acc_w), four chunks at a time with all
// their loads in flight together and a running maximum; the warps' results
// are then combined in shared memory.  Every sum runs in a fixed order, so
// the output is bit-identical from run to run.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kHeadDimMerge = 256;

// WPR warps per row: 1 (a CTA of four warps takes four rows, a warp per
// row), or 2 / 4 / 8 (a CTA per row; warp w takes slots w, w + WPR, ...).
// RUNS: the slots are the pair's runs (their count is read first) rather
// than its chunks (loaded at once, masked by the list length when it comes).
template <int WPR, bool RUNS>
__global__ void __launch_bounds__(WPR == 1 ? 128 : WPR * 32) qsa_merge_kernel(const Params p)
{
    constexpr int kWarps = WPR == 1 ? 4 : WPR;
    constexpr int kRound = 4; // chunks per warp with all loads in flight together
    __shared__ float s_acc[WPR == 1 ? 1 : WPR][kHeadDimMerge];
    __shared__ float s_m[kWarps], s_l[kWarps];
    const int lane = threadIdx.x & 31;
    const int w = WPR == 1 ? 0 : threadIdx.x >> 5; // this warp's first chunk
    const int r = WPR == 1 ? blockIdx.x * 4 + (threadIdx.x >> 5) : blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    // the next call's first kernel may launch now (it waits for this grid
    // before it reads or writes anything)
    cudaTriggerProgrammaticLaunchCompletion();
    // launched as a programmatic dependent of the chunk kernel: wait until
    // that grid has finished and its partials are visible
    cudaGridDependencySynchronize();
    if (r >= p.R) return;
    if (p.q_limit && g == 0 && threadIdx.x % (32 * (WPR == 1 ? 1 : WPR)) == 0 && r % p.H == 0) {
        // causal limits must not decrease along the window
        const int t = r / p.H;
        if (t + 1 < p.T && __ldg(p.q_limit + (size_t)b * p.T + t) > __ldg(p.q_limit + (size_t)b * p.T + t + 1))
            raise_status(p, QSA_STATUS_BAD_LIMITS);
    }
    const size_t base = ((size_t)b * p.G + g) * p.n_chunks * p.R + r;
    const size_t stride = (size_t)p.R; // chunk stride of m and l
    // a round: kRound slots per warp, every load issued together (with a
    // slot per chunk the list length is only needed to mask them, so its
    // read overlaps the loads), then folded in with a running maximum
    int start, n;
    seq_range(p, b, &start, &n);
    // slots that may be loaded: every chunk slot, or the pair's runs
    const int lim = !RUNS ? p.n_chunks
                    : n > 0 ? min(max(p.part_runs[(size_t)b * p.G + g], 0), p.n_chunks) : 0;
    float M = -INFINITY, Lpart = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c0 = w; c0 < lim; c0 += kRound * WPR) {
        float mu[kRound], lu[kRound];
        float4 ou[kRound][2];
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
            const int c = c0 + u * WPR;
            mu[u] = -INFINITY;
            lu[u] = 0.f;
            if (c < lim) {
                const size_t idx = base + (size_t)c * stride;
                mu[u] = p.part_m[idx];
                lu[u] = p.part_l[idx];
                const float4 *src = reinterpret_cast<const float4 *>(p.part_o + idx * kHeadDim + lane * 8);
                ou[u][0] = src[0];
                ou[u][1] = src[1];
            }
        }
        const int n_chunks = RUNS ? lim : n > 0 ? (n + p.chunk_cells - 1) / p.chunk_cells : 0; // valid slots
        bool ok[kRound];
        float gm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
            ok[u] = c0 + u * WPR < n_chunks && lu[u] > 0.f;
            if (ok[u]) gm = fmaxf(gm, mu[u]);
        }
        if (gm > M) {
            const float f = M == -INFINITY ? 0.f : __expf(M - gm);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] *= f;
            Lpart *= f;
            M = gm;
        }
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
            if (!ok[u]) continue;
            const float wu = mu[u] == M ? 1.f : __expf(mu[u] - M);
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
        if (c0 + kRound * WPR >= n_chunks) break;
    }
    const int t = r / p.H, j = r % p.H;
    float *orow = p.out + (((size_t)b * p.T + t) * p.G * p.H + (size_t)g * p.H + j) * kHeadDim;
    if (WPR == 1) {
        float4 *dst = reinterpret_cast<float4 *>(orow + lane * 8);
        const float L = Lpart;
        if (L > 0.f) {
            const float iL = 1.f / L;
            dst[0] = make_float4(acc[0] * iL, acc[1] * iL, acc[2] * iL, acc[3] * iL);
            dst[1] = make_float4(acc[4] * iL, acc[5] * iL, acc[6] * iL, acc[7] * iL);
        } else {
            dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const int wi = WPR == 1 ? 0 : w;
    *reinterpret_cast<float4 *>(&s_acc[wi][lane * 8]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4 *>(&s_acc[wi][lane * 8 + 4]) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if (lane == 0) {
        s_m[wi] = M;
        s_l[wi] = Lpart;
    }
    __syncthreads();

    // combine the warps' results in a fixed order; each thread owns
    // dimensions threadIdx.x, threadIdx.x + blockDim.x, ...
    float Mt = -INFINITY;
#pragma unroll
    for (int x = 0; x < kWarps; ++x)
        if (s_l[x] > 0.f) Mt = fmaxf(Mt, s_m[x]);
    float fx[kWarps];
    float L = 0.f;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) {
        fx[x] = 0.f;
        if (Mt > -INFINITY && s_l[x] > 0.f) {
            fx[x] = s_m[x] == Mt ? 1.f : __expf(s_m[x] - Mt);
            L = fmaf(s_l[x], fx[x], L);
        }
    }
    const float iL = L > 0.f ? 1.f / L : 0.f;
    for (int d = threadIdx.x; d < kHeadDimMerge; d += WPR * 32) {
        float o = 0.f;
#pragma unroll
        for (int x = 0; x < kWarps; ++x)
            if (fx[x] != 0.f) o = fmaf(s_acc[x][d], fx[x], o);
        orow[d] = L > 0.f ? o * iL : 0.f;
    }
}

} // namespace

cudaError_t launch_merge(const Params &p, cudaStream_t stream)
{
    // a warp per row when rows have few slots (chunks, or the runs the chunk
    // kernel expects to form); otherwise a CTA per row: 8 warps for more than
    // 16 slots (one round of loads covers 32) while the grid stays within 32
    // warps per SM, else 4; with more rows than 4-warp CTAs fit in one wave
    // (7 per SM), 2 warps per row (1,536 rows of 17 chunks: 30.4 -> 29.4 us
    // per call).  No wider CTA: the merge runs beside
    // the next call's chunk kernel (it lets that grid launch at once), and a
    // 16-warp CTA's 32 K registers kept chunk CTAs off its SM (one pair, 17
    // chunks: 4.6 -> 3.8 us per call with 8 warps; 64 chunks: 5.8 -> 5.2)
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long rows = (long long)p.R * p.G * p.n_seq;
    const int slots = p.merge_slots > 0 ? p.merge_slots : p.n_chunks; // expected per row
    const int wpr = slots <= 4 ? 1
                    : (slots > 16 && rows * 8 <= 32ll * sms) ? 8
                    : (rows * 4 <= 28ll * sms) ? 4 : 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(wpr == 1 ? (p.R + 3) / 4 : p.R), (unsigned)p.G, (unsigned)p.n_seq);
    cfg.blockDim = dim3(wpr == 1 ? 128 : wpr * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.runs) {
        if (wpr == 1) return cudaLaunchKernelEx(&cfg, qsa_merge_kernel<1, true>, p);
        if (wpr == 4) return cudaLaunchKernelEx(&cfg, qsa_merge_kernel<4, true>, p);
        if (wpr == 8) return cudaLaunchKernelEx(&cfg, qsa_merge_kernel<8, true>, p);
        return cudaLaunchKernelEx(&cfg, qsa_merge_kernel<2, true>, p);
    }
    if (wpr == 1) return cudaLaunchKernelEx(&cfg, qsa_merge_kernel<1, false>, p);
    if (wpr == 4) return cudaLaunchKernelEx(&cfg, qsa_merge_kernel<4, false>, p);
    if (wpr == 8) return cudaLaunchKernelEx(&cfg, qsa_merge_kernel<8, false>, p);
    return cudaLaunchKernelEx(&cfg, qsa_merge_kernel<2, false>, p);
}

} // namespace qsa
