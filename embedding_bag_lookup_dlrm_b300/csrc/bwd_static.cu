// bwd_static.cu -- the training step without a caller-provided workspace.
//
// Some callers of this library cannot allocate device memory at the point
// where they run a training step: a plugin reached through a plain C
// interface that is handed only its input and output buffers, with no
// allocator or workspace; or a process whose device memory belongs to
// another framework's pooled allocator, where a raw cudaMalloc would fail
// or fragment that pool, and where cudaMalloc / cudaFree would also stall
// the device at an unpredictable moment.  For them this file keeps the
// scratch memory of dlrm_sparse_bwd_adagrad in one fixed-size device array
// that lives as long as the library is loaded, and passes its address as
// the workspace.  Nothing here allocates.
//
// The array is shared by every call on a device and keeps what the last
// call left in it.  The training step writes every scratch byte before it
// reads it (dP, the sort keys and values, the digit counts, the partial
// sums), so nothing has to be cleared between calls.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) use the same bytes at once and race; the caller must order them.
#include <cuda_runtime.h>

#include "dlrm_sparse.h"

namespace {

constexpr size_t kScratchBytes = DLRM_STATIC_SCRATCH_BYTES;

// The scratch itself.  In host code `g_scratch` names a host-side stand-in,
// not device memory: only the address from cudaGetSymbolAddress may be
// handed to a kernel.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Address of g_scratch on the current device.  Looked up on every call (a
// cheap query once the module is loaded), never cached: after a context reset
// the array lives at a new address.
dlrm_status scratch_address(void** out)
{
    void* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_scratch) != cudaSuccess || ptr == nullptr) return DLRM_ERR_CUDA;
    *out = ptr;
    return DLRM_OK;
}

}  // namespace

extern "C" dlrm_status dlrm_sparse_bwd_adagrad_static(const dlrm_tables* tables, const dlrm_bags* bags,
                                                      dlrm_pool_mode mode, const float* dense,
                                                      const float* pooled_saved, const float* grad_out,
                                                      float* grad_dense, float* const* accum, float lr, float eps,
                                                      int32_t* status_dev, cudaStream_t stream)
{
    size_t need = 0;
    dlrm_status st = dlrm_sparse_bwd_workspace_size(tables, bags, &need);
    if (st != DLRM_OK) return st;
    if (need > kScratchBytes) return DLRM_ERR_INVALID_ARG;  // batch too large for the fixed scratch
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != DLRM_OK) return st;
    return dlrm_sparse_bwd_adagrad(tables, bags, mode, dense, pooled_saved, grad_out, grad_dense, accum, lr, eps,
                                   scratch, kScratchBytes, status_dev, stream, nullptr);
}
