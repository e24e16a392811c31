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

// The embedding-bag lookup alone (embbag.cu): a group of lanes per bag.
dlrm_status launch_embbag(const FwdArgs& args, int dim, int dtype, int index_type, cudaStream_t stream);

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
    int32_t rule;      // DLRM_RULE_ADAGRAD or DLRM_RULE_SGD
    uint64_t t_magic;  // ceil(2^64 / T) for T >= 2: sort value v = b*T + t gives b = high word of v * t_magic
};

// Where the gradient of the pooled vectors comes from.
enum BwdSource : int {
    kFromInteraction = 0,  // the interaction backward of this call (dense, pooled, grad_out)
    kFromPooledGrad = 1,   // the caller's grad_pooled [B][T][D]
};

// Workspace bytes of the training step (source kFromInteraction) or of the row
// update from a given pooled gradient (kFromPooledGrad, mean pooling needs a
// scaled copy of it).
size_t bwd_workspace_bytes(int64_t B, int32_t T, int32_t D, int64_t nnz, int source, bool mean);

// side: a second stream for the key build and sort (nullptr or == stream: one stream).
// grad_pooled: the source of kFromPooledGrad (ignored otherwise).
// presorted: the workspace holds the sorted lookups of these bags from launch_sort (side is then unused);
// sorted, if given, is an event the per-row sums wait for (the interaction backward does not); grad_ready, if
// given, is recorded on `stream` once the interaction backward is queued.
dlrm_status launch_backward(const BwdArgs& args, int dim, int index_type, int source, const float* grad_pooled,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream, cudaStream_t side,
                            bool presorted = false, cudaEvent_t sorted = nullptr, cudaEvent_t grad_ready = nullptr);

// The lookup keys of the bags and their stable radix sort into a training-step workspace (the layout
// launch_backward with source kFromInteraction reads), on `stream`.
dlrm_status launch_sort(const BwdArgs& args, int dim, int index_type, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

// The interaction backward alone: grad_dense and grad_pooled (not scaled by bag lengths).
dlrm_status launch_interact_backward(const BwdArgs& args, int dim, float* grad_pooled, cudaStream_t stream);

// Raw IDs to rows: rows[p] = raw[p] mod V_t (unsigned), t the table holding position p.
struct HashArgs {
    uint64_t num_rows[DLRM_MAX_TABLES];
    uint64_t magic[DLRM_MAX_TABLES];  // floor((2^64 - 1) / V_t)
    const uint64_t* raw;
    const void* offsets;
    void* rows;
    int32_t* status;
    int64_t B;
    int64_t nnz;
    int32_t T;
};
dlrm_status launch_hash(const HashArgs& args, int index_type, cudaStream_t stream);

// The exchange of pooled vectors between G table shards and H sample shards.
struct ExchangeArgs {
    float* by_table[DLRM_MAX_SHARDS];   // table shard g: batch x shard_tables[g] x D
    float* by_sample[DLRM_MAX_SHARDS];  // sample shard h: (sample_start[h+1] - sample_start[h]) x T x D
    int64_t sample_start[DLRM_MAX_SHARDS + 1];
    int32_t table_shard[DLRM_MAX_TABLES];
    int32_t table_slot[DLRM_MAX_TABLES];
    int32_t shard_tables[DLRM_MAX_SHARDS];
    int64_t batch;
    int32_t T, G, H, D;
    int32_t to_sample;  // 1: by_table -> by_sample, 0: by_sample -> by_table
};
dlrm_status launch_exchange(const ExchangeArgs& args, cudaStream_t stream);

// Tables in host memory with a device cache: the staging of a batch's lookups.
struct TierArgs {
    const void* host[DLRM_MAX_TABLES];  // device-readable addresses of the host tables
    void* cache[DLRM_MAX_TABLES];       // device: (C_t + M_t) rows
    const int32_t* slot_of[DLRM_MAX_TABLES];
    int64_t num_rows[DLRM_MAX_TABLES];
    int64_t cache_rows[DLRM_MAX_TABLES];
    int64_t stage_rows[DLRM_MAX_TABLES];
    const void* indices;
    const void* offsets;
    int32_t* counters;  // T staging counters (zeroed by the launch)
    int32_t* status;
    int64_t B;
    int64_t nnz;
    int32_t T;
    int32_t row_bytes;
};
dlrm_status launch_tier_stage(const TierArgs& args, int index_type, void* out, cudaStream_t stream);
dlrm_status launch_tier_fill(const void* host, void* cache, int32_t* slot_of, int64_t* slot_row, const int64_t* rows,
                             int64_t n, int64_t C, int64_t V, int row_bytes, int32_t* status, cudaStream_t stream);
dlrm_status launch_tier_init(int32_t* slot_of, int64_t V, int64_t* slot_row, int64_t C, cudaStream_t stream);

// Dense layers (mlp.cu): y = act(x W^T + b) on the tensor cores, its backward with SGD, the sigmoid head.
size_t fc_fwd_workspace_bytes(int64_t M, int32_t K, int32_t N);
dlrm_status launch_fc_fwd(const float* x, const float* w, const float* b, int64_t M, int32_t K, int32_t N, int relu,
                          float* y, void* workspace, int32_t* status, cudaStream_t stream);
size_t fc_bwd_workspace_bytes(int64_t M, int32_t K, int32_t N);
dlrm_status launch_fc_bwd_sgd(const float* x, float* w, float* b, const float* y, const float* dy, int64_t M, int32_t K,
                              int32_t N, int relu, float lr, float* dx, void* workspace, int32_t* status,
                              cudaStream_t stream);
size_t head_workspace_bytes(int64_t M, int32_t K);
dlrm_status launch_head(const float* h, float* w, float* b, const float* label, int64_t M, int32_t K, float lr,
                        float* prob, float* loss, float* dh, void* workspace, cudaStream_t stream);

}  // namespace dlrm
