// gdn_noalloc.cu -- gdn_chunk_fwd_noalloc: the chunked forward for callers
// that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory at call time: code that
// runs inside a host that forbids cudaMalloc after start-up (allocation
// would break its memory accounting or stall other streams), runtimes whose
// device memory is managed by someone else, or plug-ins that only ever get
// input and output pointers. This entry point needs nothing but those:
// its scratch is a fixed buffer compiled into the library.
//
// The buffer is a file-scope __device__ array of GDN_NOALLOC_SCRATCH_BYTES
// bytes. Every GPU that loads this part of the library holds it until the
// process exits. In host code the array's name only denotes a host-side
// shadow, so the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
gdn_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_noalloc(
    const void *q, const void *k, gdn_tensor_desc qkd, const void *v, gdn_tensor_desc vd,
    const float *g, const float *gk, const float *beta, const float *h0,
    const int32_t *cu_seqlens, int n_seq, void *out, gdn_tensor_desc od, float *h_final,
    float *den_out, int B, int T, int H, int K, int V, int chunk, int reverse, int flags,
    cudaStream_t stream) {
    // gdn_chunk_fwd's own argument checks first: given no workspace it
    // launches nothing and returns GDN_ERR_WORKSPACE exactly when every
    // argument check passed, so a bad argument gets the status gdn_chunk_fwd
    // would give it
    const gdn_status pre = gdn_chunk_fwd(q, k, qkd, v, vd, g, gk, beta, h0, cu_seqlens, n_seq, out,
                                         od, h_final, den_out, B, T, H, K, V, chunk, reverse, flags,
                                         nullptr, 0, stream);
    if (pre != GDN_ERR_WORKSPACE) return pre;
    const size_t need = gdn_workspace_size(B, T, H, K, V, n_seq, cu_seqlens != nullptr,
                                           qkd.dtype, den_out != nullptr);
    if (need == 0 || need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    void *scratch = nullptr;
    const gdn_status st = scratch_address(&scratch);
    if (st != GDN_OK) return st;
    return gdn_chunk_fwd(q, k, qkd, v, vd, g, gk, beta, h0, cu_seqlens, n_seq, out, od, h_final,
                         den_out, B, T, H, K, V, chunk, reverse, flags, scratch,
                         (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}

// The error word sits at the start of the built-in buffer, where
// gdn_chunk_fwd keeps it in any workspace.
extern "C" gdn_status gdn_noalloc_last_device_error(cudaStream_t stream, int *word) {
    void *scratch = nullptr;
    const gdn_status st = scratch_address(&scratch);
    if (st != GDN_OK) return st;
    return gdn_last_device_error(scratch, stream, word);
}
