// api.cu -- the C ABI declared in include/dlrm_sparse.h: host-side argument
// checks, packing of the kernel parameter blocks, launches.  Nothing here
// allocates device memory or touches data on the host.
#include <stdint.h>
#include <string.h>

#include "dlrm_sparse.h"
#include "internal.h"

namespace {

using dlrm::BwdArgs;
using dlrm::FwdArgs;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dim_supported(int32_t D) { return D == 16 || D == 32 || D == 64 || D == 128 || D == 256; }

dlrm_status check_tables(const dlrm_tables* t)
{
    if (t == nullptr || t->data == nullptr || t->num_rows == nullptr) return DLRM_ERR_INVALID_ARG;
    if (t->num_tables < 1 || t->num_tables > DLRM_MAX_TABLES) return DLRM_ERR_INVALID_ARG;
    if (t->dtype != DLRM_F32 && t->dtype != DLRM_BF16) return DLRM_ERR_INVALID_ARG;
    if (t->dim <= 0 || t->dim > 256 || t->dim % 4 != 0) return DLRM_ERR_INVALID_ARG;
    if (!dim_supported(t->dim)) return DLRM_ERR_UNSUPPORTED;
    for (int i = 0; i < t->num_tables; ++i) {
        if (t->data[i] == nullptr || !aligned16(t->data[i])) return DLRM_ERR_INVALID_ARG;
        if (t->num_rows[i] < 1) return DLRM_ERR_INVALID_ARG;
    }
    return DLRM_OK;
}

dlrm_status check_bags(const dlrm_bags* b, int32_t T)
{
    if (b == nullptr || b->batch < 1 || b->nnz < 0) return DLRM_ERR_INVALID_ARG;
    if (b->index_type != DLRM_I32 && b->index_type != DLRM_I64) return DLRM_ERR_INVALID_ARG;
    if (b->offsets == nullptr || (b->nnz > 0 && b->indices == nullptr)) return DLRM_ERR_INVALID_ARG;
    if (b->batch > (int64_t{1} << 40) / T) return DLRM_ERR_INVALID_ARG;
    if (b->index_type == DLRM_I32 && (b->nnz > INT32_MAX || int64_t{T} * b->batch + 1 > INT32_MAX))
        return DLRM_ERR_INVALID_ARG;
    return DLRM_OK;
}

bool mode_ok(dlrm_pool_mode m) { return m == DLRM_POOL_SUM || m == DLRM_POOL_MEAN; }

// The forward kernels count a warp's or a bag's lookups in 32-bit integers.
dlrm_status check_forward_size(const dlrm_bags* b)
{
    return b->nnz > INT32_MAX ? DLRM_ERR_UNSUPPORTED : DLRM_OK;
}

void pack_forward(FwdArgs& a, const dlrm_tables* t, const dlrm_bags* b, dlrm_pool_mode mode)
{
    memset(&a, 0, sizeof a);
    for (int i = 0; i < t->num_tables; ++i) {
        a.tables[i] = t->data[i];
        a.num_rows[i] = t->num_rows[i];
    }
    a.indices = b->indices;
    a.offsets = b->offsets;
    a.B = b->batch;
    a.nnz = b->nnz;
    a.T = t->num_tables;
    a.mean = mode == DLRM_POOL_MEAN;
}

int64_t out_width(int32_t T, int32_t D) { return D + int64_t{T + 1} * T / 2; }

}  // namespace

extern "C" {

int32_t dlrm_abi_version(void) { return 2; }

const char* dlrm_status_string(dlrm_status s)
{
    if (s == DLRM_OK) return "ok";
    if (s & DLRM_ERR_INVALID_ARG) return "invalid argument";
    if (s & DLRM_ERR_INDEX_OOB) return "index out of range";
    if (s & DLRM_ERR_BAD_OFFSETS) return "malformed offsets";
    if (s & DLRM_ERR_TIMEOUT) return "device wait timed out";
    if (s & DLRM_ERR_CUDA) return "CUDA error";
    if (s & DLRM_ERR_UNSUPPORTED) return "unsupported configuration";
    if (s & DLRM_ERR_CAPACITY) return "staging capacity exceeded";
    return "unknown status";
}

dlrm_status dlrm_embbag_fwd(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode, float* pooled,
                            int32_t* status_dev, cudaStream_t stream)
{
    dlrm_status st = check_tables(tables);
    if (st != DLRM_OK) return st;
    if ((st = check_bags(bags, tables->num_tables)) != DLRM_OK) return st;
    if (!mode_ok(mode) || pooled == nullptr || !aligned16(pooled)) return DLRM_ERR_INVALID_ARG;
    if ((st = check_forward_size(bags)) != DLRM_OK) return st;
    FwdArgs a;
    pack_forward(a, tables, bags, mode);
    a.pooled_out = pooled;
    a.status = status_dev;
    return dlrm::launch_forward(dlrm::kEmbbag, a, tables->dim, tables->dtype, bags->index_type, stream);
}

dlrm_status dlrm_interact_fwd(const float* dense, const float* pooled, int64_t batch, int32_t num_tables, int32_t dim,
                              float* out, cudaStream_t stream)
{
    if (dense == nullptr || pooled == nullptr || out == nullptr) return DLRM_ERR_INVALID_ARG;
    if (!aligned16(dense) || !aligned16(pooled) || (reinterpret_cast<uintptr_t>(out) & 3u)) return DLRM_ERR_INVALID_ARG;
    if (batch < 1 || num_tables < 1 || num_tables > DLRM_MAX_TABLES) return DLRM_ERR_INVALID_ARG;
    if (dim <= 0 || dim > 256 || dim % 4 != 0) return DLRM_ERR_INVALID_ARG;
    if (!dim_supported(dim)) return DLRM_ERR_UNSUPPORTED;
    FwdArgs a;
    memset(&a, 0, sizeof a);
    a.dense = dense;
    a.pooled_in = pooled;
    a.out = out;
    a.B = batch;
    a.T = num_tables;
    return dlrm::launch_forward(dlrm::kInteract, a, dim, DLRM_F32, DLRM_I32, stream);
}

dlrm_status dlrm_sparse_fwd(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode, const float* dense,
                            float* out, float* pooled_save, int32_t* status_dev, cudaStream_t stream)
{
    dlrm_status st = check_tables(tables);
    if (st != DLRM_OK) return st;
    if ((st = check_bags(bags, tables->num_tables)) != DLRM_OK) return st;
    if (!mode_ok(mode) || dense == nullptr || out == nullptr || !aligned16(dense)) return DLRM_ERR_INVALID_ARG;
    if ((st = check_forward_size(bags)) != DLRM_OK) return st;
    if (reinterpret_cast<uintptr_t>(out) & 3u) return DLRM_ERR_INVALID_ARG;
    if (pooled_save != nullptr && !aligned16(pooled_save)) return DLRM_ERR_INVALID_ARG;
    FwdArgs a;
    pack_forward(a, tables, bags, mode);
    a.dense = dense;
    a.out = out;
    a.pooled_out = pooled_save;
    a.status = status_dev;
    return dlrm::launch_forward(dlrm::kFused, a, tables->dim, tables->dtype, bags->index_type, stream);
}

dlrm_status dlrm_sparse_fwd_host(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode,
                                 const float* dense_host, float* out_host, void* indices_dev, void* offsets_dev,
                                 float* dense_dev, float* out_dev, int32_t* status_dev, cudaStream_t stream)
{
    dlrm_status st = check_tables(tables);
    if (st != DLRM_OK) return st;
    if ((st = check_bags(bags, tables->num_tables)) != DLRM_OK) return st;
    if (dense_host == nullptr || out_host == nullptr || offsets_dev == nullptr || dense_dev == nullptr ||
        out_dev == nullptr || (bags->nnz > 0 && indices_dev == nullptr))
        return DLRM_ERR_INVALID_ARG;
    const size_t isz = bags->index_type == DLRM_I32 ? 4 : 8;
    const int64_t B = bags->batch, T = tables->num_tables, D = tables->dim;
    if (bags->nnz > 0 &&
        cudaMemcpyAsync(indices_dev, bags->indices, bags->nnz * isz, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return DLRM_ERR_CUDA;
    if (cudaMemcpyAsync(offsets_dev, bags->offsets, (T * B + 1) * isz, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return DLRM_ERR_CUDA;
    if (cudaMemcpyAsync(dense_dev, dense_host, B * D * sizeof(float), cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return DLRM_ERR_CUDA;
    dlrm_bags dev = *bags;
    dev.indices = indices_dev;
    dev.offsets = offsets_dev;
    st = dlrm_sparse_fwd(tables, &dev, mode, dense_dev, out_dev, nullptr, status_dev, stream);
    if (st != DLRM_OK) return st;
    const size_t out_bytes = static_cast<size_t>(B) * out_width(tables->num_tables, tables->dim) * sizeof(float);
    if (cudaMemcpyAsync(out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return DLRM_ERR_CUDA;
    return DLRM_OK;
}

dlrm_status dlrm_sparse_bwd_workspace_size(const dlrm_tables* tables, const dlrm_bags* bags, size_t* bytes)
{
    dlrm_status st = check_tables(tables);
    if (st != DLRM_OK) return st;
    if ((st = check_bags(bags, tables->num_tables)) != DLRM_OK) return st;
    if (bytes == nullptr) return DLRM_ERR_INVALID_ARG;
    *bytes = dlrm::bwd_workspace_bytes(bags->batch, tables->num_tables, tables->dim, bags->nnz, dlrm::kFromInteraction,
                                       true);
    return DLRM_OK;
}

dlrm_status dlrm_embbag_bwd_workspace_size(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode,
                                           size_t* bytes)
{
    dlrm_status st = check_tables(tables);
    if (st != DLRM_OK) return st;
    if ((st = check_bags(bags, tables->num_tables)) != DLRM_OK) return st;
    if (bytes == nullptr || !mode_ok(mode)) return DLRM_ERR_INVALID_ARG;
    *bytes = dlrm::bwd_workspace_bytes(bags->batch, tables->num_tables, tables->dim, bags->nnz, dlrm::kFromPooledGrad,
                                       mode == DLRM_POOL_MEAN);
    return DLRM_OK;
}

}  // extern "C"

namespace {

// The 32-bit limits of the sort and the parameters the lookup keys need
// (tables, row counts and bases, bags); checked tables and bags.
dlrm_status pack_rows(BwdArgs& a, const dlrm_tables* tables, const dlrm_bags* bags, int32_t* status_dev)
{
    int64_t total_rows = 0;
    for (int i = 0; i < tables->num_tables; ++i) total_rows += tables->num_rows[i];
    // 32-bit sort keys (global row ids, the sentinel 2^32 - 1 above them), 32-bit sort values (dP row
    // b*T + t) and 32-bit positions in the sorted lookups
    if (total_rows >= (int64_t{1} << 32) - 1) return DLRM_ERR_UNSUPPORTED;
    if (int64_t{tables->num_tables} * bags->batch >= (int64_t{1} << 32)) return DLRM_ERR_UNSUPPORTED;
    if (bags->nnz >= (int64_t{1} << 32)) return DLRM_ERR_UNSUPPORTED;
    memset(&a, 0, sizeof a);
    int64_t base = 0;
    for (int i = 0; i < tables->num_tables; ++i) {
        a.tables[i] = static_cast<float*>(tables->data[i]);
        a.num_rows[i] = tables->num_rows[i];
        a.row_base[i] = base;
        base += tables->num_rows[i];
    }
    a.row_base[tables->num_tables] = base;
    a.indices = bags->indices;
    a.offsets = bags->offsets;
    a.status = status_dev;
    a.B = bags->batch;
    a.nnz = bags->nnz;
    a.T = tables->num_tables;
    a.t_magic = a.T >= 2 ? ~uint64_t{0} / static_cast<uint64_t>(a.T) + 1 : 0;
    return DLRM_OK;
}

// Checks shared by the row-update entry points; fills everything of the
// parameter block but the interaction inputs.
dlrm_status pack_update(BwdArgs& a, const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode,
                        const dlrm_update* upd, void* workspace, int32_t* status_dev)
{
    dlrm_status st = check_tables(tables);
    if (st != DLRM_OK) return st;
    if ((st = check_bags(bags, tables->num_tables)) != DLRM_OK) return st;
    if (tables->dtype != DLRM_F32) return DLRM_ERR_UNSUPPORTED;
    if (!mode_ok(mode) || upd == nullptr || workspace == nullptr || !aligned16(workspace)) return DLRM_ERR_INVALID_ARG;
    if (upd->rule != DLRM_RULE_ADAGRAD && upd->rule != DLRM_RULE_SGD) return DLRM_ERR_INVALID_ARG;
    if (upd->rule == DLRM_RULE_ADAGRAD && upd->accum == nullptr) return DLRM_ERR_INVALID_ARG;
    if ((st = pack_rows(a, tables, bags, status_dev)) != DLRM_OK) return st;
    for (int i = 0; i < tables->num_tables; ++i) {
        if (upd->rule == DLRM_RULE_ADAGRAD) {
            if (upd->accum[i] == nullptr || !aligned16(upd->accum[i])) return DLRM_ERR_INVALID_ARG;
            a.accum[i] = upd->accum[i];
        }
    }
    a.mean = mode == DLRM_POOL_MEAN;
    a.lr = upd->lr;
    a.eps = upd->eps;
    a.rule = upd->rule;
    return DLRM_OK;
}

// The training step; presorted: the workspace holds the sorted lookups of these bags (dlrm_sparse_bwd_sort).
dlrm_status sparse_bwd(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode, const float* dense,
                       const float* pooled_saved, const float* grad_out, float* grad_dense, const dlrm_update* update,
                       void* workspace, size_t workspace_bytes, int32_t* status_dev, cudaStream_t stream,
                       cudaStream_t side_stream, bool presorted, cudaEvent_t sorted, cudaEvent_t grad_ready)
{
    BwdArgs a;
    dlrm_status st = pack_update(a, tables, bags, mode, update, workspace, status_dev);
    if (st != DLRM_OK) return st;
    if (dense == nullptr || pooled_saved == nullptr || grad_out == nullptr || grad_dense == nullptr)
        return DLRM_ERR_INVALID_ARG;
    if (!aligned16(dense) || !aligned16(pooled_saved) || !aligned16(grad_dense) ||
        (reinterpret_cast<uintptr_t>(grad_out) & 3u))
        return DLRM_ERR_INVALID_ARG;
    if (workspace_bytes < dlrm::bwd_workspace_bytes(bags->batch, tables->num_tables, tables->dim, bags->nnz,
                                                    dlrm::kFromInteraction, true))
        return DLRM_ERR_INVALID_ARG;
    a.dense = dense;
    a.pooled = pooled_saved;
    a.grad_out = grad_out;
    a.grad_dense = grad_dense;
    return dlrm::launch_backward(a, tables->dim, bags->index_type, dlrm::kFromInteraction, nullptr, workspace,
                                 workspace_bytes, stream, side_stream, presorted, sorted, grad_ready);
}

}  // namespace

extern "C" {

dlrm_status dlrm_sparse_bwd_update(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode,
                                   const float* dense, const float* pooled_saved, const float* grad_out,
                                   float* grad_dense, const dlrm_update* update, void* workspace,
                                   size_t workspace_bytes, int32_t* status_dev, cudaStream_t stream,
                                   cudaStream_t side_stream)
{
    return sparse_bwd(tables, bags, mode, dense, pooled_saved, grad_out, grad_dense, update, workspace,
                      workspace_bytes, status_dev, stream, side_stream, false, nullptr, nullptr);
}

dlrm_status dlrm_sparse_bwd_sort(const dlrm_tables* tables, const dlrm_bags* bags, void* workspace,
                                 size_t workspace_bytes, int32_t* status_dev, cudaStream_t stream)
{
    dlrm_status st = check_tables(tables);
    if (st != DLRM_OK) return st;
    if ((st = check_bags(bags, tables->num_tables)) != DLRM_OK) return st;
    if (tables->dtype != DLRM_F32) return DLRM_ERR_UNSUPPORTED;
    if (workspace == nullptr || !aligned16(workspace)) return DLRM_ERR_INVALID_ARG;
    BwdArgs a;
    if ((st = pack_rows(a, tables, bags, status_dev)) != DLRM_OK) return st;
    if (workspace_bytes < dlrm::bwd_workspace_bytes(bags->batch, tables->num_tables, tables->dim, bags->nnz,
                                                    dlrm::kFromInteraction, true))
        return DLRM_ERR_INVALID_ARG;
    return dlrm::launch_sort(a, tables->dim, bags->index_type, workspace, workspace_bytes, stream);
}

dlrm_status dlrm_sparse_bwd_update_sorted(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode,
                                          const float* dense, const float* pooled_saved, const float* grad_out,
                                          float* grad_dense, const dlrm_update* update, void* workspace,
                                          size_t workspace_bytes, int32_t* status_dev, cudaEvent_t sorted,
                                          cudaEvent_t grad_ready, cudaStream_t stream)
{
    return sparse_bwd(tables, bags, mode, dense, pooled_saved, grad_out, grad_dense, update, workspace,
                      workspace_bytes, status_dev, stream, nullptr, true, sorted, grad_ready);
}

dlrm_status dlrm_sparse_bwd_adagrad(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode,
                                    const float* dense, const float* pooled_saved, const float* grad_out,
                                    float* grad_dense, float* const* accum, float lr, float eps, void* workspace,
                                    size_t workspace_bytes, int32_t* status_dev, cudaStream_t stream,
                                    cudaStream_t side_stream)
{
    if (accum == nullptr) return DLRM_ERR_INVALID_ARG;
    const dlrm_update upd = {DLRM_RULE_ADAGRAD, lr, eps, accum};
    return dlrm_sparse_bwd_update(tables, bags, mode, dense, pooled_saved, grad_out, grad_dense, &upd, workspace,
                                  workspace_bytes, status_dev, stream, side_stream);
}

dlrm_status dlrm_embbag_bwd_update(const dlrm_tables* tables, const dlrm_bags* bags, dlrm_pool_mode mode,
                                   const float* grad_pooled, const dlrm_update* update, void* workspace,
                                   size_t workspace_bytes, int32_t* status_dev, cudaStream_t stream,
                                   cudaStream_t side_stream)
{
    BwdArgs a;
    dlrm_status st = pack_update(a, tables, bags, mode, update, workspace, status_dev);
    if (st != DLRM_OK) return st;
    if (grad_pooled == nullptr || !aligned16(grad_pooled)) return DLRM_ERR_INVALID_ARG;
    if (workspace_bytes < dlrm::bwd_workspace_bytes(bags->batch, tables->num_tables, tables->dim, bags->nnz,
                                                    dlrm::kFromPooledGrad, mode == DLRM_POOL_MEAN))
        return DLRM_ERR_INVALID_ARG;
    return dlrm::launch_backward(a, tables->dim, bags->index_type, dlrm::kFromPooledGrad, grad_pooled, workspace,
                                 workspace_bytes, stream, side_stream);
}

dlrm_status dlrm_interact_bwd(const float* dense, const float* pooled, const float* grad_out, int64_t batch,
                              int32_t num_tables, int32_t dim, float* grad_dense, float* grad_pooled,
                              cudaStream_t stream)
{
    if (dense == nullptr || pooled == nullptr || grad_out == nullptr || grad_dense == nullptr ||
        grad_pooled == nullptr)
        return DLRM_ERR_INVALID_ARG;
    if (!aligned16(dense) || !aligned16(pooled) || !aligned16(grad_dense) || !aligned16(grad_pooled) ||
        (reinterpret_cast<uintptr_t>(grad_out) & 3u))
        return DLRM_ERR_INVALID_ARG;
    if (batch < 1 || batch > (int64_t{1} << 40) || num_tables < 1 || num_tables > DLRM_MAX_TABLES)
        return DLRM_ERR_INVALID_ARG;
    if (dim <= 0 || dim > 256 || dim % 4 != 0) return DLRM_ERR_INVALID_ARG;
    if (!dim_supported(dim)) return DLRM_ERR_UNSUPPORTED;
    BwdArgs a;
    memset(&a, 0, sizeof a);
    a.dense = dense;
    a.pooled = pooled;
    a.grad_out = grad_out;
    a.grad_dense = grad_dense;
    a.B = batch;
    a.T = num_tables;
    return dlrm::launch_interact_backward(a, dim, grad_pooled, stream);
}

dlrm_status dlrm_pooled_exchange(const dlrm_shard_plan* plan, float* const* by_table, float* const* by_sample,
                                 int32_t to_sample, cudaStream_t stream)
{
    if (plan == nullptr || by_table == nullptr || by_sample == nullptr) return DLRM_ERR_INVALID_ARG;
    const int G = plan->num_table_shards, H = plan->num_sample_shards, T = plan->num_tables, D = plan->dim;
    if (G < 1 || G > DLRM_MAX_SHARDS || H < 1 || H > DLRM_MAX_SHARDS || T < 1 || T > DLRM_MAX_TABLES)
        return DLRM_ERR_INVALID_ARG;
    if (plan->batch < 1 || plan->batch > (int64_t{1} << 40) / T) return DLRM_ERR_INVALID_ARG;
    if (plan->table_shard == nullptr || plan->table_slot == nullptr || plan->sample_start == nullptr)
        return DLRM_ERR_INVALID_ARG;
    if (D <= 0 || D > 256 || D % 4 != 0) return DLRM_ERR_INVALID_ARG;
    if (!dim_supported(D)) return DLRM_ERR_UNSUPPORTED;
    if (to_sample != 0 && to_sample != 1) return DLRM_ERR_INVALID_ARG;
    dlrm::ExchangeArgs a;
    memset(&a, 0, sizeof a);
    // every shard's slots are 0 .. T_g - 1, each once
    bool seen[DLRM_MAX_TABLES] = {};
    for (int t = 0; t < T; ++t) {
        const int g = plan->table_shard[t];
        if (g < 0 || g >= G) return DLRM_ERR_INVALID_ARG;
        a.table_shard[t] = g;
        a.shard_tables[g] += 1;
    }
    for (int g = 0; g < G; ++g) {
        for (int k = 0; k < T; ++k) seen[k] = false;
        for (int t = 0; t < T; ++t) {
            if (plan->table_shard[t] != g) continue;
            const int slot = plan->table_slot[t];
            if (slot < 0 || slot >= a.shard_tables[g] || seen[slot]) return DLRM_ERR_INVALID_ARG;
            seen[slot] = true;
            a.table_slot[t] = slot;
        }
        if (a.shard_tables[g] > 0 && (by_table[g] == nullptr || !aligned16(by_table[g]))) return DLRM_ERR_INVALID_ARG;
        a.by_table[g] = by_table[g];
    }
    if (plan->sample_start[0] != 0 || plan->sample_start[H] != plan->batch) return DLRM_ERR_INVALID_ARG;
    for (int h = 0; h < H; ++h) {
        const int64_t n = plan->sample_start[h + 1] - plan->sample_start[h];
        if (n < 0) return DLRM_ERR_INVALID_ARG;
        if (n > 0 && (by_sample[h] == nullptr || !aligned16(by_sample[h]))) return DLRM_ERR_INVALID_ARG;
        a.by_sample[h] = by_sample[h];
        a.sample_start[h] = plan->sample_start[h];
    }
    a.sample_start[H] = plan->batch;
    a.batch = plan->batch;
    a.T = T;
    a.G = G;
    a.H = H;
    a.D = D;
    a.to_sample = to_sample;
    return dlrm::launch_exchange(a, stream);
}

}  // extern "C"

namespace {

dlrm_status check_tiered(const dlrm_tiered_tables* t)
{
    if (t == nullptr || t->host_data == nullptr || t->num_rows == nullptr || t->slot_of == nullptr ||
        t->slot_row == nullptr || t->cache == nullptr || t->cache_rows == nullptr || t->stage_rows == nullptr)
        return DLRM_ERR_INVALID_ARG;
    if (t->num_tables < 1 || t->num_tables > DLRM_MAX_TABLES) return DLRM_ERR_INVALID_ARG;
    if (t->dtype != DLRM_F32 && t->dtype != DLRM_BF16) return DLRM_ERR_INVALID_ARG;
    if (t->dim <= 0 || t->dim > 256 || t->dim % 4 != 0) return DLRM_ERR_INVALID_ARG;
    if (!dim_supported(t->dim)) return DLRM_ERR_UNSUPPORTED;
    for (int i = 0; i < t->num_tables; ++i) {
        if (t->num_rows[i] < 1 || t->cache_rows[i] < 0 || t->stage_rows[i] < 0) return DLRM_ERR_INVALID_ARG;
        if (t->cache_rows[i] + t->stage_rows[i] > INT32_MAX) return DLRM_ERR_UNSUPPORTED;  // 32-bit slots
        if (t->host_data[i] == nullptr || !aligned16(t->host_data[i]) || t->slot_of[i] == nullptr) return DLRM_ERR_INVALID_ARG;
        if (t->cache_rows[i] + t->stage_rows[i] > 0 && (t->cache[i] == nullptr || !aligned16(t->cache[i])))
            return DLRM_ERR_INVALID_ARG;
        if (t->cache_rows[i] > 0 && t->slot_row[i] == nullptr) return DLRM_ERR_INVALID_ARG;
    }
    return DLRM_OK;
}

int row_bytes_of(const dlrm_tiered_tables* t) { return t->dim * (t->dtype == DLRM_F32 ? 4 : 2); }

}  // namespace

extern "C" {

dlrm_status dlrm_tier_init(const dlrm_tiered_tables* tables, cudaStream_t stream)
{
    dlrm_status st = check_tiered(tables);
    if (st != DLRM_OK) return st;
    for (int t = 0; t < tables->num_tables; ++t) {
        st = dlrm::launch_tier_init(tables->slot_of[t], tables->num_rows[t], tables->slot_row[t],
                                    tables->cache_rows[t], stream);
        if (st != DLRM_OK) return st;
    }
    return DLRM_OK;
}

dlrm_status dlrm_tier_cache_fill(const dlrm_tiered_tables* tables, int32_t table, const int64_t* rows, int64_t n,
                                 int32_t* status_dev, cudaStream_t stream)
{
    dlrm_status st = check_tiered(tables);
    if (st != DLRM_OK) return st;
    if (table < 0 || table >= tables->num_tables || n < 0 || n > tables->cache_rows[table] ||
        (n > 0 && rows == nullptr))
        return DLRM_ERR_INVALID_ARG;
    return dlrm::launch_tier_fill(tables->host_data[table], tables->cache[table], tables->slot_of[table],
                                  tables->slot_row[table], rows, n, tables->cache_rows[table], tables->num_rows[table],
                                  row_bytes_of(tables), status_dev, stream);
}

dlrm_status dlrm_tier_stage(const dlrm_tiered_tables* tables, const dlrm_bags* bags, void* indices_out,
                            int32_t* counters, int32_t* status_dev, cudaStream_t stream)
{
    dlrm_status st = check_tiered(tables);
    if (st != DLRM_OK) return st;
    if ((st = check_bags(bags, tables->num_tables)) != DLRM_OK) return st;
    if (counters == nullptr || (bags->nnz > 0 && indices_out == nullptr)) return DLRM_ERR_INVALID_ARG;
    dlrm::TierArgs a;
    memset(&a, 0, sizeof a);
    for (int t = 0; t < tables->num_tables; ++t) {
        a.host[t] = tables->host_data[t];
        a.cache[t] = tables->cache[t];
        a.slot_of[t] = tables->slot_of[t];
        a.num_rows[t] = tables->num_rows[t];
        a.cache_rows[t] = tables->cache_rows[t];
        a.stage_rows[t] = tables->stage_rows[t];
    }
    a.indices = bags->indices;
    a.offsets = bags->offsets;
    a.counters = counters;
    a.status = status_dev;
    a.B = bags->batch;
    a.nnz = bags->nnz;
    a.T = tables->num_tables;
    a.row_bytes = row_bytes_of(tables);
    return dlrm::launch_tier_stage(a, bags->index_type, indices_out, stream);
}

}  // extern "C"

namespace {

bool fc_dims_ok(int64_t batch, int32_t in_dim, int32_t out_dim)
{
    return batch >= 1 && batch < (int64_t{1} << 31) && in_dim >= 1 && in_dim <= 65536 && out_dim >= 1 &&
           out_dim <= 65536;
}

}  // namespace

extern "C" {

dlrm_status dlrm_fc_fwd_workspace_size(int64_t batch, int32_t in_dim, int32_t out_dim, size_t* bytes)
{
    if (bytes == nullptr || !fc_dims_ok(batch, in_dim, out_dim)) return DLRM_ERR_INVALID_ARG;
    *bytes = dlrm::fc_fwd_workspace_bytes(batch, in_dim, out_dim);
    return DLRM_OK;
}

dlrm_status dlrm_fc_fwd(const float* x, const float* w, const float* b, int64_t batch, int32_t in_dim,
                        int32_t out_dim, int32_t act, float* y, void* workspace, size_t workspace_bytes,
                        int32_t* status_dev, cudaStream_t stream)
{
    if (x == nullptr || w == nullptr || y == nullptr || workspace == nullptr || !fc_dims_ok(batch, in_dim, out_dim))
        return DLRM_ERR_INVALID_ARG;
    if (act != DLRM_ACT_NONE && act != DLRM_ACT_RELU) return DLRM_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(workspace) || (b != nullptr && !aligned16(b)))
        return DLRM_ERR_INVALID_ARG;
    if (workspace_bytes < dlrm::fc_fwd_workspace_bytes(batch, in_dim, out_dim)) return DLRM_ERR_INVALID_ARG;
    return dlrm::launch_fc_fwd(x, w, b, batch, in_dim, out_dim, act == DLRM_ACT_RELU, y, workspace, status_dev, stream);
}

dlrm_status dlrm_fc_bwd_workspace_size(int64_t batch, int32_t in_dim, int32_t out_dim, size_t* bytes)
{
    if (bytes == nullptr || !fc_dims_ok(batch, in_dim, out_dim)) return DLRM_ERR_INVALID_ARG;
    *bytes = dlrm::fc_bwd_workspace_bytes(batch, in_dim, out_dim);
    return DLRM_OK;
}

dlrm_status dlrm_fc_bwd_sgd(const float* x, float* w, float* b, const float* y, const float* dy, int64_t batch,
                            int32_t in_dim, int32_t out_dim, int32_t act, float lr, float* dx, void* workspace,
                            size_t workspace_bytes, int32_t* status_dev, cudaStream_t stream)
{
    if (x == nullptr || w == nullptr || dy == nullptr || workspace == nullptr || !fc_dims_ok(batch, in_dim, out_dim))
        return DLRM_ERR_INVALID_ARG;
    if (act != DLRM_ACT_NONE && act != DLRM_ACT_RELU) return DLRM_ERR_INVALID_ARG;
    if (act == DLRM_ACT_RELU && y == nullptr) return DLRM_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(dy) || !aligned16(workspace) || (y != nullptr && !aligned16(y)) ||
        (dx != nullptr && !aligned16(dx)) || (b != nullptr && !aligned16(b)))
        return DLRM_ERR_INVALID_ARG;
    if (workspace_bytes < dlrm::fc_bwd_workspace_bytes(batch, in_dim, out_dim)) return DLRM_ERR_INVALID_ARG;
    return dlrm::launch_fc_bwd_sgd(x, w, b, y, dy, batch, in_dim, out_dim, act == DLRM_ACT_RELU, lr, dx, workspace,
                                   status_dev, stream);
}

dlrm_status dlrm_head_bce_workspace_size(int64_t batch, int32_t in_dim, size_t* bytes)
{
    if (bytes == nullptr || batch < 1 || batch > (int64_t{1} << 31) || in_dim < 1) return DLRM_ERR_INVALID_ARG;
    if (in_dim > 1024) return DLRM_ERR_UNSUPPORTED;
    *bytes = dlrm::head_workspace_bytes(batch, in_dim);
    return DLRM_OK;
}

dlrm_status dlrm_head_bce_sgd(const float* h, float* w, float* b, const float* label, int64_t batch, int32_t in_dim,
                              float lr, float* prob, float* loss, float* dh, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream)
{
    if (h == nullptr || w == nullptr || b == nullptr || label == nullptr || dh == nullptr || workspace == nullptr)
        return DLRM_ERR_INVALID_ARG;
    size_t need = 0;
    dlrm_status st = dlrm_head_bce_workspace_size(batch, in_dim, &need);
    if (st != DLRM_OK) return st;
    if (workspace_bytes < need || !aligned16(workspace)) return DLRM_ERR_INVALID_ARG;
    return dlrm::launch_head(h, w, b, label, batch, in_dim, lr, prob, loss, dh, workspace, stream);
}

dlrm_status dlrm_hash_indices(const int64_t* num_rows, int32_t num_tables, int64_t batch, int64_t nnz,
                              const uint64_t* raw_ids, const void* offsets, int32_t index_type, void* rows,
                              int32_t* status_dev, cudaStream_t stream)
{
    if (num_rows == nullptr || offsets == nullptr || num_tables < 1 || num_tables > DLRM_MAX_TABLES)
        return DLRM_ERR_INVALID_ARG;
    if (batch < 1 || nnz < 0 || batch > (int64_t{1} << 40) / num_tables) return DLRM_ERR_INVALID_ARG;
    if (nnz > 0 && (raw_ids == nullptr || rows == nullptr)) return DLRM_ERR_INVALID_ARG;
    if (index_type != DLRM_I32 && index_type != DLRM_I64) return DLRM_ERR_INVALID_ARG;
    if (index_type == DLRM_I32 && (nnz > INT32_MAX || int64_t{num_tables} * batch + 1 > INT32_MAX))
        return DLRM_ERR_INVALID_ARG;
    dlrm::HashArgs a;
    memset(&a, 0, sizeof a);
    for (int t = 0; t < num_tables; ++t) {
        if (num_rows[t] < 1) return DLRM_ERR_INVALID_ARG;
        if (index_type == DLRM_I32 && num_rows[t] > int64_t{INT32_MAX} + 1) return DLRM_ERR_INVALID_ARG;
        a.num_rows[t] = static_cast<uint64_t>(num_rows[t]);
        a.magic[t] = ~uint64_t{0} / a.num_rows[t];
    }
    a.raw = raw_ids;
    a.offsets = offsets;
    a.rows = rows;
    a.status = status_dev;
    a.B = batch;
    a.nnz = nnz;
    a.T = num_tables;
    return dlrm::launch_hash(a, index_type, stream);
}

}  // extern "C"
