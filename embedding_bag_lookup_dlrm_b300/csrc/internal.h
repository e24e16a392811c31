// internal.h -- launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

#include "dlrm_sparse.h"

namespace dlrm {

enum FwdMode : int {
    kEmbbag = 0,    // gather + pool, write pooled
    kFused = 1,     // gather + pool + interaction, write out (and pooled if asked)
    kInteract = 2,  // interaction of given dense + pooled, write out
};

// Everything a forward kernel needs, passed by value as one kernel parameter.
struct FwdArgs {
    const void* tables[DLRM_MAX_TABLES];
    int64_t num_rows[DLRM_MAX_TABLES];
    const void* indices;
    const void* offsets;
    const float* dense;
    const float* pooled_in;
    float* out;
    float* pooled_out;
    int32_t* status;
    int64_t B;
    int64_t nnz;
    int32_t T;
    int32_t mean;
};

// Number of SMs of the current device (0 on error).
int sm_count();
// Registers per thread of a compiled kernel (0 on error).
int kernel_registers(const void* kernel);

// Launch one forward pass.  dim in {16,32,64,128,256}; dtype/index_type as in
// the ABI.  Returns DLRM_OK, DLRM_ERR_UNSUPPORTED or DLRM_ERR_CUDA.
dlrm_status launch_forward(int mode, const FwdArgs& args, int dim, int dtype, int index_type,
                           cudaStream_t stream);

// The same forward with the interaction on the tensor cores (fwd_tc.cu):
// fused and interaction modes, D in {64, 128}, N = T + 1 <= 128, bags of
// at most two lookups on average.
bool forward_tc_supported(int mode, int dim, int num_tables, int64_t batch, int64_t nnz);
dlrm_status launch_forward_tc(int mode, const FwdArgs& args, int dim, int dtype, int index_type,
                              cudaStream_t stream);

// ---- training step -------------------------------------------------------
struct BwdArgs {
    float* tables[DLRM_MAX_TABLES];
    float* accum[DLRM_MAX_TABLES];
    int64_t num_rows[DLRM_MAX_TABLES];
    int64_t row_base[DLRM_MAX_TABLES + 1];  // prefix sum of num_rows
    const void* indices;
    const void* offsets;
    const float* dense;
    const float* pooled;
    const float* grad_out;
    float* grad_dense;
    int32_t* status;
    int64_t B;
    int64_t nnz;
    int32_t T;
    int32_t mean;
    float lr;
    float eps;
    uint64_t t_magic;  // ceil(2^64 / T) for T >= 2: sort value v = b*T + t gives b = high word of v * t_magic
};

size_t bwd_workspace_bytes(int64_t B, int32_t T, int32_t D, int64_t nnz);

// side: a second stream for the key build and sort (nullptr or == stream: one stream).
dlrm_status launch_backward(const BwdArgs& args, int dim, int index_type, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream, cudaStream_t side);

}  // namespace dlrm
