// qsa_noalloc.cu -- qsa_decode_attn_step_noalloc: the single-sequence call
// with the library's own fixed scratch buffer in place of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory where they run
// decode attention -- a runtime whose memory budget is fixed after start-up
// (no allocator call may happen on the serving path), a plugin embedded in a
// host application that owns all device memory and exposes no allocator, or
// code that must not touch an allocator at all.  Such a caller still owns
// the inputs and the output; only the chunk partials (the scratch) move into
// a file-scope __device__ array that lives in every GPU that loads this
// library, until the process exits.
//
// The array's name is only a host-side stand-in in host code, so the device
// address is looked up with cudaGetSymbolAddress, with the device current.  A
// symbol's address belongs to the CUDA context it was loaded into, so a call
// on a stream that is not being captured looks it up again (a cheap call that
// allocates nothing) and refreshes the per-device copy; a call made while its
// stream is being captured into a CUDA graph uses that copy, so the first
// call on each device, and the first after a cudaDeviceReset or a switch of
// context, must happen outside capture.
//
// Every call shares the one array and leaves its contents behind; the chunk
// kernels write every partial the merge reads, so nothing needs clearing.
// Calls whose kernels overlap on the GPU (for example on two streams) race
// on the array and must be serialised by the caller.
#include <mutex>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20; // 8 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device: looked up
// afresh unless the stream is being captured, when the copy from the last
// lookup on this device is used.
qsa_status scratch_address(cudaStream_t stream, void **addr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return QSA_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return QSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return QSA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    } else if (g_scratch_addr[dev] == nullptr) {
        return QSA_ERR_CUDA; // first call on this device inside a capture
    }
    *addr = g_scratch_addr[dev];
    return QSA_OK;
}

} // namespace
} // namespace qsa

extern "C" qsa_status qsa_decode_attn_step_noalloc(const qsa_shape *shape, const void *q,
                                                   const int8_t *k_pool, const int8_t *v_pool,
                                                   const float *k_scale, const float *v_scale,
                                                   const int32_t *page_table, const int32_t *sel,
                                                   int32_t n_sel, float *out, uint32_t *status,
                                                   void *stream)
{
    if (n_sel < 0) return QSA_ERR_INVALID_ARG;
    size_t need = 0;
    qsa_status st = qsa_workspace_bytes(shape, 1, n_sel, &need);
    if (st != QSA_OK) return st;
    if (need > qsa::kNoAllocScratchBytes) return QSA_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = qsa::scratch_address(static_cast<cudaStream_t>(stream), &scratch);
    if (st != QSA_OK) return st;
    return qsa_decode_attn_step(shape, q, k_pool, v_pool, k_scale, v_scale, page_table, sel,
                                n_sel, out, scratch, qsa::kNoAllocScratchBytes, status, stream);
}
