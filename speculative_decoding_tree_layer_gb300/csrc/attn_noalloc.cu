// attn_noalloc.cu -- dflv_tree_attn_verify_noalloc: the attention tree verify
// for callers that cannot allocate device memory themselves (see
// include/dflv.h).  Its merge scratch is one fixed array in the library's own
// device memory instead of a caller-provided workspace.
//
// In host code the name g_attn_scratch stands for a host-side shadow, not for
// a device address: the address the kernels need is fetched once per device
// with cudaGetSymbolAddress (with that device current) and then reused.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "../../include/dflv.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = (size_t)DFLV_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "the scratch keeps 256-byte granules");

// One scratch area per device that loads the library, held until exit.
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices];  // device address of g_attn_scratch, per device (null: not yet fetched)

// The scratch's device address on the current device; fetched on the first
// call per device.
dflv_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DFLV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DFLV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();  // leave no sticky error for the caller's next CUDA call
            return DFLV_ERR_CUDA;
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return DFLV_OK;
}

}  // namespace

extern "C" dflv_status dflv_tree_attn_verify_noalloc(const dflv_attn_desc* desc, const int32_t* parent,
                                                     const int32_t* n_nodes, const int32_t* n_past,
                                                     const uint16_t* q, const uint16_t* k_new,
                                                     const uint16_t* v_new, const dflv_kv_layer* cache,
                                                     float* out, int32_t* status_dev, dflv_stream_t stream) {
    // a shape whose merge needs more than the fixed scratch is refused before
    // anything is launched
    if (dflv_attn_workspace_size(desc) > kScratchBytes) return DFLV_ERR_CAPACITY;
    void* ws = nullptr;
    const dflv_status s = scratch_address(&ws);
    if (s != DFLV_OK) return s;
    return dflv_tree_attn_verify(desc, parent, n_nodes, n_past, q, k_new, v_new, cache, out, status_dev, ws,
                                 kScratchBytes, stream);
}
