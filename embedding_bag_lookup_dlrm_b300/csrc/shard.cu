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
// HBM-bound: each row is read once and written once.  One warp per row, the
// rows in sample-major order so that consecutive warps write (or read)
// consecutive rows of a by-sample buffer.
#include "common.cuh"
#include "internal.h"

namespace dlrm {
namespace {

constexpr int kExThreads = 256;

__global__ void __launch_bounds__(kExThreads) exchange_kernel(const __grid_constant__ ExchangeArgs a)
{
    const int lane = threadIdx.x % kWarp;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kExThreads / kWarp);
    const int64_t rows = a.batch * a.T;
    const int chunks = a.D / 4;
    for (int64_t r = blockIdx.x * int64_t{kExThreads / kWarp} + threadIdx.x / kWarp; r < rows; r += warps) {
        const int64_t b = r / a.T;
        const int t = static_cast<int>(r - b * a.T);
        int lo = 0, hi = a.H - 1;  // the sample shard of b: the last h with sample_start[h] <= b
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.sample_start[mid] <= b)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int g = a.table_shard[t];
        float4* tp = reinterpret_cast<float4*>(a.by_table[g] + (b * a.shard_tables[g] + a.table_slot[t]) * a.D);
        float4* sp = reinterpret_cast<float4*>(a.by_sample[lo] + ((b - a.sample_start[lo]) * a.T + t) * a.D);
        if (a.to_sample) {
            for (int c = lane; c < chunks; c += kWarp) sp[c] = tp[c];
        } else {
            for (int c = lane; c < chunks; c += kWarp) tp[c] = sp[c];
        }
    }
}

}  // namespace

dlrm_status launch_exchange(const ExchangeArgs& a, cudaStream_t s)
{
    const int64_t rows = a.batch * a.T;
    if (rows == 0) return DLRM_OK;
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    const int64_t want = (rows + kExThreads / kWarp - 1) / (kExThreads / kWarp);
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    exchange_kernel<<<static_cast<unsigned>(want < cap ? want : cap), kExThreads, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

}  // namespace dlrm
