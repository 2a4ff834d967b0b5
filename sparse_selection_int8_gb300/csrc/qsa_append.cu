// qsa_append.cu -- qsa_kv_append: new K and V rows quantised to INT8 codes
// with one fp32 scale per (cell, KV head), written into the pools at the
// slots the page table gives for the cells' logical positions.
//
// The step is the KV append that follows the K/V projections of a QSA layer
// ("Strata issue #8, round 9: performance candidate set on v0.2.9",
// R9-gpu-8, implementation handoff); what it writes is the format the decode-attention
// step reads ("attn_chunk_q8_v3_kernel": INT8 K/V pools with per-cell fp32
// scales).  The pages print no quantiser; the reading here is the plainest
// symmetric one: scale = max|x| / 127, code = x / scale rounded to nearest,
// ties to even, both in fp32 (correctly rounded divisions), a zero row gets
// scale 0 and zero codes.
//
// HBM-bound: per new cell and KV head it reads the K and V rows (2 x 1 KB of
// fp32, or 2 x 512 B of bf16) and writes 2 x 256 code bytes and two scales.
// One warp per new cell (sequence, cell) with all its KV heads: lane l holds
// elements 8l..8l+7 of a row (each warp load is 1 KB or 512 B of contiguous
// memory), the row maximum is one warp reduction, and lane l stores its 8
// codes as one 8-byte word (256 contiguous bytes per warp store).  The row
// loads do not depend on the page-table lookup, so they are issued first and
// overlap it; the rows of two KV heads are in flight at once.  Codes come
// from correctly rounded quotients (remainder-corrected reciprocals, below)
// rounded half to even by the 1.5 * 2^23 addition, a few instructions per
// element.  Grid: as many blocks of 8 warps as are resident at once, striding
// over the new cells.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kAppendWarps = 8;
constexpr int kAppendThreads = kAppendWarps * 32;

struct AppendParams {
    const void *k_new, *v_new; // [n_seq][n_new][G][D]
    const int32_t *positions;  // [n_seq][n_new]
    const int32_t *page_table; // [n_seq][page_table_len]
    int8_t *k_pool, *v_pool;   // [n_seq][G][pool_cells][D]
    float *k_scale, *v_scale;  // [n_seq][G][pool_cells]
    uint32_t *status;
    uint32_t pairs;            // n_seq * n_new (new cells); pairs * G < 2^31
    uint32_t n_new, G;
    int pool_cells, page_table_len;
    int page_cells, pool_pages; // P cells per page; valid page entries 0 .. pool_pages - 1
    int bf16;
};

// The raw 16-byte pieces of one lane's 8 elements of a row: two for fp32,
// one for bf16 (the other unused).
struct Raw8 {
    uint4 a, b;
};

template <bool BF16>
__device__ __forceinline__ Raw8 load_raw8(const void *base, uint32_t row, int lane)
{
    Raw8 r;
    if (BF16) {
        r.a = ldg_nc_v4(static_cast<const uint8_t *>(base) + (size_t)row * kHeadDim * 2 + 16 * lane);
        r.b = make_uint4(0u, 0u, 0u, 0u);
    } else {
        const uint8_t *p = static_cast<const uint8_t *>(base) + (size_t)row * kHeadDim * 4 + 32 * lane;
        r.a = ldg_nc_v4(p);
        r.b = ldg_nc_v4(p + 16);
    }
    return r;
}

template <bool BF16>
__device__ __forceinline__ void widen8(const Raw8 &r, float *x)
{
    if (BF16) {
        const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = bf16_bits_to_f32(w[k] & 0xffffu);
            x[2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
        }
    } else {
        const uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = __uint_as_float(w[k]);
    }
}

// a / b correctly rounded, given yb = RN(1/b), for normal a, b with a/b
// normal and far from overflow, by remainder corrections (Markstein's method,
// as given in Muller et al., "Handbook of Floating-Point Arithmetic",
// division by Newton-Raphson iteration with FMA): q + (a - q b) yb equals
// a/b + (1 - b yb)(q - a/b), so the first correction brings RN(a yb) within
// one ulp of a/b, where the remainder a - q b is exact in one FMA and the
// second correction rounds correctly.  Five instructions.  (Here a quotient
// below the normal range is a code of 0 whichever way its last bits fall.)
__device__ __forceinline__ float div_rn_by(float a, float b, float yb)
{
    float q = a * yb;
    float r = fmaf(-q, b, a);
    q = fmaf(r, yb, q);
    r = fmaf(-q, b, a);
    return fmaf(r, yb, q);
}

// For |q| <= 127.5: the int8 code of q rounded to the nearest integer, ties
// to even, in the low byte.  The fp32 sum q + 1.5 * 2^23 lies in [2^23, 2^24),
// where the unit in the last place is 1, so the addition rounds q half to
// even and the low mantissa bits hold 0x400000 + rint(q).
__device__ __forceinline__ uint32_t rint_low_byte(float q)
{
    return __float_as_uint(__fadd_rn(q, 12582912.f));
}

// Codes of this lane's 8 elements (packed little-endian) and the row scale.
__device__ __forceinline__ uint2 quantize8(const float *x, float &scale)
{
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(x[k]));
    // non-negative floats order like their bit patterns
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
    if (!(amax > 0.f)) {
        scale = 0.f;
        return make_uint2(0u, 0u);
    }
    uint32_t c[8];
    if (amax >= 0x1p-90f) { // the same for the whole warp
        scale = div_rn_by(amax, 127.f, 1.f / 127.f);
        const float y = __frcp_rn(scale);
#pragma unroll
        for (int k = 0; k < 8; ++k) c[k] = rint_low_byte(div_rn_by(x[k], scale, y));
    } else { // tiny rows: plain correctly rounded divisions
        scale = __fdiv_rn(amax, 127.f);
#pragma unroll
        for (int k = 0; k < 8; ++k) c[k] = rint_low_byte(__fdiv_rn(x[k], scale));
    }
    // |code| <= 127 (x / scale <= 127 up to rounding), so the low bytes are
    // the int8 codes
    return make_uint2(__byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410),
                      __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410));
}

// One quantised (cell, KV head): both rows' codes and scales to the pools.
template <bool BF16>
__device__ __forceinline__ void store_item(const AppendParams &p, const Raw8 &kr, const Raw8 &vr,
                                           size_t cell, int lane)
{
    float x[8], ks, vs;
    widen8<BF16>(kr, x);
    const uint2 kc = quantize8(x, ks);
    widen8<BF16>(vr, x);
    const uint2 vc = quantize8(x, vs);
    *reinterpret_cast<uint2 *>(p.k_pool + cell * kHeadDim + 8 * lane) = kc;
    *reinterpret_cast<uint2 *>(p.v_pool + cell * kHeadDim + 8 * lane) = vc;
    if (lane == 0) {
        p.k_scale[cell] = ks;
        p.v_scale[cell] = vs;
    }
}

// A warp per new cell (sequence b, cell i) at a time, all its KV heads: the
// position and page entry are looked up once, and the rows of two heads are
// loaded before the lookup's result is needed.
template <bool BF16>
__global__ void __launch_bounds__(kAppendThreads, 4) qsa_kv_append_kernel(const AppendParams p)
{
    const int lane = threadIdx.x & 31;
    const uint32_t warps = gridDim.x * kAppendWarps;
    for (uint32_t bi = blockIdx.x * kAppendWarps + (threadIdx.x >> 5); bi < p.pairs; bi += warps) {
        const uint32_t row0 = bi * p.G; // row of head 0 in the new K/V arrays
        Raw8 k0 = load_raw8<BF16>(p.k_new, row0, lane), v0 = load_raw8<BF16>(p.v_new, row0, lane);
        Raw8 k1{}, v1{};
        if (p.G > 1) {
            k1 = load_raw8<BF16>(p.k_new, row0 + 1, lane);
            v1 = load_raw8<BF16>(p.v_new, row0 + 1, lane);
        }
        const int pos = __ldg(p.positions + bi);
        const uint32_t b = bi / p.n_new;
        // position pos: page pos / P at offset pos % P; the entry is a page of the pool
        const int P = p.page_cells;
        int slot = -1;
        uint32_t bad = 0;
        if (pos < 0 || (long long)pos >= (long long)p.page_table_len * P) {
            bad = QSA_STATUS_BAD_POSITION;
        } else {
            const int page = P == 1 ? pos : pos / P;
            const int e = __ldg(p.page_table + (size_t)b * p.page_table_len + page);
            if (e == -1) bad = QSA_STATUS_NOT_RESIDENT;
            else if (e < 0 || e >= p.pool_pages) bad = QSA_STATUS_BAD_SLOT;
            else slot = P == 1 ? e : e * P + (pos - page * P);
        }
        if (bad) { // the whole warp agrees
            if (lane == 0 && p.status) atomicOr(p.status, bad);
            continue;
        }
        const size_t cell0 = (size_t)b * p.G * p.pool_cells + slot; // head g: + g * pool_cells
        for (uint32_t g = 0; g < p.G; g += 2) {
            if (g > 0) {
                k0 = load_raw8<BF16>(p.k_new, row0 + g, lane);
                v0 = load_raw8<BF16>(p.v_new, row0 + g, lane);
                if (g + 1 < p.G) {
                    k1 = load_raw8<BF16>(p.k_new, row0 + g + 1, lane);
                    v1 = load_raw8<BF16>(p.v_new, row0 + g + 1, lane);
                }
            }
            store_item<BF16>(p, k0, v0, cell0 + (size_t)g * p.pool_cells, lane);
            if (g + 1 < p.G) store_item<BF16>(p, k1, v1, cell0 + (size_t)(g + 1) * p.pool_cells, lane);
        }
    }
}

bool aligned(const void *ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

} // namespace
} // namespace qsa

extern "C" qsa_status qsa_kv_append(const qsa_shape *shape, int32_t n_seq, int32_t n_new,
                                    int32_t kv_dtype, const void *k_new, const void *v_new,
                                    const int32_t *positions, const int32_t *page_table,
                                    int8_t *k_pool, int8_t *v_pool, float *k_scale,
                                    float *v_scale, uint32_t *status, void *stream)
{
    using qsa::aligned;
    if (!shape) return QSA_ERR_INVALID_ARG;
    if (shape->n_kv_heads < 1 || shape->pool_cells < 1 || shape->page_table_len < 1)
        return QSA_ERR_INVALID_ARG;
    if (shape->head_dim != qsa::kHeadDim) return QSA_ERR_UNSUPPORTED;
    if (shape->page_cells < 0) return QSA_ERR_INVALID_ARG;
    const int P = shape->page_cells > 0 ? shape->page_cells : 1;
    if (shape->pool_cells % P != 0 || (long long)shape->page_table_len * P > 0x7fffffffll)
        return QSA_ERR_INVALID_ARG;
    if (n_seq < 0 || n_new < 0) return QSA_ERR_INVALID_ARG;
    if (kv_dtype != QSA_F32 && kv_dtype != QSA_BF16) return QSA_ERR_INVALID_ARG;
    if (!k_new || !v_new || !positions || !page_table || !k_pool || !v_pool || !k_scale || !v_scale)
        return QSA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(positions, 4) ||
        !aligned(page_table, 4) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(k_scale, 4) || !aligned(v_scale, 4) || (status && !aligned(status, 4)))
        return QSA_ERR_INVALID_ARG;
    if ((const void *)k_pool == k_new || (const void *)k_pool == v_new ||
        (const void *)v_pool == k_new || (const void *)v_pool == v_new || k_pool == v_pool ||
        k_scale == v_scale)
        return QSA_ERR_INVALID_ARG;
    const long long items = (long long)n_seq * n_new * shape->n_kv_heads;
    if (items == 0) return QSA_OK;
    if (items >= (1ll << 31)) return QSA_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QSA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QSA_ERR_CUDA;
    qsa::AppendParams p{};
    p.k_new = k_new;
    p.v_new = v_new;
    p.positions = positions;
    p.page_table = page_table;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.status = status;
    p.pairs = (uint32_t)((long long)n_seq * n_new);
    p.n_new = (uint32_t)n_new;
    p.G = (uint32_t)shape->n_kv_heads;
    p.pool_cells = shape->pool_cells;
    p.page_table_len = shape->page_table_len;
    p.page_cells = P;
    p.pool_pages = shape->pool_cells / P;
    p.bf16 = kv_dtype == QSA_BF16;
    // as many blocks as are resident at once (every warp strides over items)
    auto kernel = p.bf16 ? qsa::qsa_kv_append_kernel<true> : qsa::qsa_kv_append_kernel<false>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, qsa::kAppendThreads, 0) != cudaSuccess)
        return QSA_ERR_CUDA;
    const long long blocks_needed = ((long long)p.pairs + qsa::kAppendWarps - 1) / qsa::kAppendWarps;
    const long long cap = (long long)sms * (per_sm > 0 ? per_sm : 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(blocks_needed < cap ? blocks_needed : cap));
    cfg.blockDim = dim3(qsa::kAppendThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    return cudaLaunchKernelEx(&cfg, kernel, p) == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
