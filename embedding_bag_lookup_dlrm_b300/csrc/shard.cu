// shard.cu -- the exchange of pooled vectors in a table-wise model-parallel
// step ("DLRM", robocikowo.com: embedding tables split across devices, model
// parallel, with an all-to-all of the lookup results before the interaction
// layer; "DLRM explained", "How do you size compute for a DLRM...": tables
// sharded, NCCL all-to-all).
//
// Table shard g owns T_g tables and pools them for every sample of the batch:
// by_table[g] is B x T_g x D.  Sample shard h owns the samples
// [s_h, s_{h+1}) and needs all T pooled vectors of them for the interaction:
// by_sample[h] is (s_{h+1} - s_h) x T x D.  The exchange copies every
// (sample, table) row from one layout to the other (forward), or back
// (backward, the gradients of the pooled vectors).  With every shard on this
// device it is the whole all-to-all; after a collective all-to-all between
// devices (each receiving, from every table shard, the rows of its own
// samples) it is the local unpack, with one sample shard.
//
// HBM-bound: each row is read once and written once.  A warp moves one sample
// at a time: its T rows are one contiguous block of the by-sample buffer, and
// row t of it sits in the by-table buffer of t's owner at sample stride
// T_g * D.  The block stages, per table, that source (or destination) base and
// stride in shared memory; a lane then walks the sample's T*D/4 16-byte chunks
// (consecutive lanes, consecutive chunks) with kUnroll loads in flight before
// the matching stores.
#include "common.cuh"
#include "internal.h"

namespace dlrm {
namespace {

constexpr int kExThreads = 256;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kExThreads) exchange_kernel(const __grid_constant__ ExchangeArgs a, int chunk_shift)
{
    __shared__ float* tab_base[DLRM_MAX_TABLES];   // by_table[g] + slot(t) * D
    __shared__ int64_t tab_stride[DLRM_MAX_TABLES];  // T_g * D: elements between samples
    __shared__ int64_t start[DLRM_MAX_SHARDS + 1];
    for (int t = threadIdx.x; t < a.T; t += kExThreads) {
        const int g = a.table_shard[t];
        tab_base[t] = a.by_table[g] + static_cast<int64_t>(a.table_slot[t]) * a.D;
        tab_stride[t] = static_cast<int64_t>(a.shard_tables[g]) * a.D;
    }
    for (int h = threadIdx.x; h <= a.H; h += kExThreads) start[h] = a.sample_start[h];
    __syncthreads();

    const int lane = threadIdx.x % kWarp;
    const int chunk_mask = (1 << chunk_shift) - 1;  // 16-byte chunks per row: D / 4, a power of two
    const int n = a.T << chunk_shift;                // chunks per sample
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kExThreads / kWarp);
    for (int64_t b = blockIdx.x * int64_t{kExThreads / kWarp} + threadIdx.x / kWarp; b < a.batch; b += warps) {
        int lo = 0, hi = a.H - 1;  // the sample shard of b: the last h with start[h] <= b
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (start[mid] <= b)
                lo = mid;
            else
                hi = mid - 1;
        }
        float4* sample_side = reinterpret_cast<float4*>(a.by_sample[lo] + (b - start[lo]) * a.T * a.D);
        for (int e0 = 0; e0 < n; e0 += kUnroll * kWarp) {
            float4 v[kUnroll];
            float4* far[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int e = e0 + u * kWarp + lane;
                far[u] = nullptr;
                if (e < n) {
                    const int t = e >> chunk_shift;
                    far[u] = reinterpret_cast<float4*>(tab_base[t] + b * tab_stride[t]) + (e & chunk_mask);
                    v[u] = a.to_sample ? *far[u] : sample_side[e];
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int e = e0 + u * kWarp + lane;
                if (e < n) {
                    if (a.to_sample)
                        sample_side[e] = v[u];
                    else
                        *far[u] = v[u];
                }
            }
        }
    }
}

}  // namespace

dlrm_status launch_exchange(const ExchangeArgs& a, cudaStream_t s)
{
    if (a.batch == 0) return DLRM_OK;
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    int chunk_shift = 0;
    while ((1 << chunk_shift) < a.D / 4) ++chunk_shift;
    if ((1 << chunk_shift) != a.D / 4) return DLRM_ERR_UNSUPPORTED;
    const int64_t want = (a.batch + kExThreads / kWarp - 1) / (kExThreads / kWarp);
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    exchange_kernel<<<static_cast<unsigned>(want < cap ? want : cap), kExThreads, 0, s>>>(a, chunk_shift);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

}  // namespace dlrm
