// noalloc.cu -- dsa_decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch on the call path: an
// engine that pre-reserves all device memory for its own pool, or code that
// must not run the device-synchronising cudaMalloc/cudaFree.  For them the
// fused step takes its scratch from one file-scope device array of fixed size
// instead of a caller workspace.  The pages have no counterpart of this entry
// point; it is an addition of this library.
#include <atomic>

#include "common.cuh"

namespace {

// The shared scratch of every dsa_decode_noalloc call on a device.  Each GPU
// that loads the library holds one copy until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// Device address of g_noalloc_scratch per device.  In host code the symbol
// itself is only a host-side stand-in and must never be handed to a kernel.
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// The device address of this device's copy of the array, looked up with the
// device current.  Outside stream capture it is looked up again on every call
// (cheap), so that a module reloaded after cudaDeviceReset is followed; while
// `stream` is capturing, the address stored by the last call outside capture
// is used, since a capture must not be disturbed.
dsa_status scratch_for_current_device(cudaStream_t stream, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return DSA_ERR_CUDA;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return DSA_ERR_CUDA;
    }
    void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (cs == cudaStreamCaptureStatusNone || p == nullptr) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_noalloc_scratch) != cudaSuccess || q == nullptr) {
            (void)cudaGetLastError();
            return DSA_ERR_CUDA;
        }
        g_scratch_ptr[dev].store(q, std::memory_order_release);
        p = q;
    }
    *out = p;
    return DSA_OK;
}

}  // namespace

extern "C" dsa_status dsa_decode_noalloc(const dsa_batch* batch, const uint8_t* q_fp8,
                                         const float* q_scale, const float* w,
                                         const void* index_pages, dsa_key_format key_format,
                                         const uint16_t* q_lat, const void* latent_pages,
                                         float kv_scale, float sm_scale, int32_t topk,
                                         uint16_t* out, float* lse, int32_t* indices,
                                         int32_t* dev_status, dsa_stream_t stream) {
    if (batch == nullptr) return DSA_ERR_INVALID_ARG;
    const size_t need = dsa_decode_workspace_size(batch, topk);
    if (need > (size_t)DSA_NOALLOC_SCRATCH_BYTES) return DSA_ERR_WORKSPACE;
    void* scratch = nullptr;
    dsa_status st = scratch_for_current_device((cudaStream_t)stream, &scratch);
    if (st != DSA_OK) return st;
    return dsa_decode(batch, q_fp8, q_scale, w, index_pages, key_format, q_lat, latent_pages,
                      kv_scale, sm_scale, topk, out, lse, indices, scratch,
                      (size_t)DSA_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
