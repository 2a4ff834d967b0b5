// qsa_chunk_simt.cu -- CUDA-core chunk kernel (steps a1-a4 on the SIMT pipes).
//
// The plain second path next to the tensor-core kernels: one CTA per (chunk,
// row block, KV head, sequence); each warp owns RPW query rows and walks the
// chunk's cells in list order with an online softmax, so each chunk partial
// is produced in one pass ("Strata PR #2220, attn_chunk_q8_v3_kernel":
// the chunk kernel reads each cell's INT8 K/V row once for all 12 heads of
// the warp's rows; lane l owns dimensions 8l..8l+7, as on the pages).
//
// Cells are staged 32 at a time: 32 threads resolve list entry -> page slot,
// then all threads copy the 32 K and V rows (256 B each) into shared memory
// with 16-byte read-only loads.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / 32;
constexpr int kStage = 32; // cells staged per step

__device__ __forceinline__ void int8x8_to_f32(uint2 raw, float *f)
{
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = (float)(int8_t)((raw.x >> (8 * e)) & 0xff);
#pragma unroll
    for (int e = 0; e < 4; ++e) f[4 + e] = (float)(int8_t)((raw.y >> (8 * e)) & 0xff);
}

template <int RPW>
__global__ void __launch_bounds__(kSimtThreads)
qsa_chunk_simt_kernel(const Params p, int n_row_blocks)
{
    __shared__ __align__(16) int8_t s_k[kStage][kHeadDim];
    __shared__ __align__(16) int8_t s_v[kStage][kHeadDim];
    __shared__ int s_slot[kStage];
    __shared__ int s_pos[kStage];
    __shared__ float s_ks[kStage];
    __shared__ float s_vs[kStage];

    cudaTriggerProgrammaticLaunchCompletion(); // the merge kernel waits for this grid anyway
    const int chunk = blockIdx.x / n_row_blocks;
    const int rb = blockIdx.x % n_row_blocks;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    int start, n;
    seq_range(p, b, &start, &n);
    const int c0 = chunk * p.chunk_cells;
    if (c0 >= n) return;
    const int c1 = (int)min((long long)c0 + p.chunk_cells, (long long)n);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int GH = p.G * p.H;
    const size_t kv_base = ((size_t)b * p.G + g) * p.pool_cells;

    float qv[RPW][8];
    bool rvalid[RPW];
    int rlim[RPW]; // causal limit of the row's query (positions below it are seen)
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = rb * kSimtWarps * RPW + warp + kSimtWarps * i;
        rvalid[i] = r < p.R;
        const int t = rvalid[i] ? r / p.H : 0, j = rvalid[i] ? r % p.H : 0;
        rlim[i] = p.q_limit ? __ldg(p.q_limit + (size_t)b * p.T + t) : INT_MAX;
        const size_t qoff = (((size_t)b * p.T + t) * GH + (size_t)g * p.H + j) * kHeadDim + lane * 8;
        if (!rvalid[i]) {
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[i][e] = 0.f;
        } else if (p.q_bf16) {
            uint4 raw = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) + qoff);
            uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qv[i][2 * e] = bf16_bits_to_f32(w[e] & 0xffff);
                qv[i][2 * e + 1] = bf16_bits_to_f32(w[e] >> 16);
            }
        } else {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(p.q) + qoff);
            float4 a = src[0], c = src[1];
            qv[i][0] = a.x; qv[i][1] = a.y; qv[i][2] = a.z; qv[i][3] = a.w;
            qv[i][4] = c.x; qv[i][5] = c.y; qv[i][6] = c.z; qv[i][7] = c.w;
        }
    }

    float m2[RPW], l[RPW], o[RPW][8];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        m2[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[i][e] = 0.f;
    }

    for (int tile = c0; tile < c1; tile += kStage) {
        const int nt = min(kStage, c1 - tile);
        __syncthreads(); // previous stage fully consumed
        if (threadIdx.x < kStage) {
            const int i = threadIdx.x;
            int slot = -1, pos = 0;
            if (i < nt) {
                pos = __ldg(p.sel + start + tile + i);
                slot = resolve_slot(p, b, pos);
            }
            s_slot[i] = slot;
            s_pos[i] = pos;
            s_ks[i] = slot >= 0 ? __ldg(p.k_scale + kv_base + slot) : 0.f;
            s_vs[i] = slot >= 0 ? __ldg(p.v_scale + kv_base + slot) : 0.f;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < 2 * kStage * 16; e += kSimtThreads) {
            const int which = e / (kStage * 16);
            const int cell = (e / 16) % kStage;
            const int piece = e % 16;
            const int slot = s_slot[cell];
            uint4 val = make_uint4(0, 0, 0, 0);
            if (slot >= 0) {
                const int8_t *src = (which ? p.v_pool : p.k_pool) + (kv_base + slot) * kHeadDim + piece * 16;
                val = ldg_nc_v4(src);
            }
            int8_t *dst = which ? &s_v[cell][piece * 16] : &s_k[cell][piece * 16];
            *reinterpret_cast<uint4 *>(dst) = val;
        }
        __syncthreads();
        for (int c = 0; c < nt; ++c) {
            if (s_slot[c] < 0) continue; // masked: uniform across the CTA
            float kf[8], vf[8];
            int8x8_to_f32(*reinterpret_cast<const uint2 *>(&s_k[c][lane * 8]), kf);
            int8x8_to_f32(*reinterpret_cast<const uint2 *>(&s_v[c][lane * 8]), vf);
            const float ksc = s_ks[c] * p.scale_log2;
            const float vsc = s_vs[c];
#pragma unroll
            for (int e = 0; e < 8; ++e) vf[e] *= vsc;
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                if (!rvalid[i] || s_pos[c] >= rlim[i]) continue; // uniform across the warp
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) dot = fmaf(qv[i][e], kf[e], dot);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
                const float s = dot * ksc;
                const float mn = fmaxf(m2[i], s);
                const float corr = fast_exp2(m2[i] - mn);
                const float pr = fast_exp2(s - mn);
                l[i] = l[i] * corr + pr;
#pragma unroll
                for (int e = 0; e < 8; ++e) o[i][e] = fmaf(o[i][e], corr, pr * vf[e]);
                m2[i] = mn;
            }
        }
    }

#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        if (!rvalid[i]) continue;
        const int r = rb * kSimtWarps * RPW + warp + kSimtWarps * i;
        const size_t idx = (((size_t)b * p.G + g) * p.n_chunks + chunk) * p.R + r;
        if (lane == 0) {
            p.part_m[idx] = m2[i] * kLn2;
            p.part_l[idx] = l[i];
        }
        float4 *dst = reinterpret_cast<float4 *>(p.part_o + idx * kHeadDim + lane * 8);
        dst[0] = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
        dst[1] = make_float4(o[i][4], o[i][5], o[i][6], o[i][7]);
    }
}

template <int RPW>
cudaError_t launch_rpw(const Params &p, cudaStream_t stream)
{
    const int rows_per_cta = kSimtWarps * RPW;
    const int n_row_blocks = (p.R + rows_per_cta - 1) / rows_per_cta;
    dim3 grid((unsigned)((long long)p.n_chunks * n_row_blocks), (unsigned)p.G, (unsigned)p.n_seq);
    qsa_chunk_simt_kernel<RPW><<<grid, kSimtThreads, 0, stream>>>(p, n_row_blocks);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_chunk_simt(const Params &p, cudaStream_t stream)
{
    if (p.n_chunks == 0) return cudaSuccess;
    const int rpw = (p.R + kSimtWarps - 1) / kSimtWarps;
    switch (rpw) {
    case 1: return launch_rpw<1>(p, stream);
    case 2: return launch_rpw<2>(p, stream);
    case 3: return launch_rpw<3>(p, stream);
    case 4: return launch_rpw<4>(p, stream);
    case 5: return launch_rpw<5>(p, stream);
    case 6: return launch_rpw<6>(p, stream);
    default: return launch_rpw<8>(p, stream);
    }
}

} // namespace qsa
