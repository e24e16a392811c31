// tier.cu -- tables larger than device memory: the rows in host memory the
// device can read, a device cache of hot rows, and a staging pre-pass that
// makes every lookup of a batch a lookup into device memory ("DLRM explained",
// "How do you size compute for a DLRM...": tables beyond device memory held in
// host RAM; "DLRM", robocikowo.com, the CPU-inference paragraph; popularity
// follows a power law, so a small set of hot rows takes most lookups).
//
// Table t keeps, in device memory, a buffer of C_t + M_t rows: slots
// [0, C_t) hold cached rows, [C_t, C_t + M_t) receive the batch's misses; and
// a map slot_of[V_t] (the slot of each row, or -1) with its inverse
// slot_row[C_t].  Staging resolves every lookup: a cached row's index becomes
// its slot; a missed row is copied from host memory into the next staging row
// (a per-table counter hands the rows out) and its index becomes that row; an
// index outside [0, V_t) becomes -1, which the forward flags and pools as
// zero, as it does for the untiered table.  The forward then runs on the
// device buffers with the rewritten indices and gives the untiered result
// bit for bit: every lookup reads a bit-exact copy of its row.
//
// A warp takes 32 consecutive lookups (one lane each for the index, the table
// search and the map), then copies the missed rows four at a time, all 32
// lanes on each row (host reads over the link, 16 bytes a lane, the four rows'
// reads in flight together).
#include "common.cuh"
#include "internal.h"

namespace dlrm {
namespace {

constexpr int kTierThreads = 256;
constexpr int kMissRows = 4;  // missed rows a warp reads from host memory at once

template <typename TI>
__global__ void __launch_bounds__(kTierThreads) stage_kernel(const __grid_constant__ TierArgs a, TI* out)
{
    __shared__ int64_t bound[DLRM_MAX_TABLES + 1];
    const TI* off = static_cast<const TI*>(a.offsets);
    const TI* ind = static_cast<const TI*>(a.indices);
    for (int t = threadIdx.x; t <= a.T; t += blockDim.x) bound[t] = static_cast<int64_t>(off[static_cast<int64_t>(t) * a.B]);
    __syncthreads();
    const int lane = threadIdx.x % kWarp;
    const int chunks = a.row_bytes / 16;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kTierThreads / kWarp);
    for (int64_t p0 = (blockIdx.x * int64_t{kTierThreads / kWarp} + threadIdx.x / kWarp) * kWarp; p0 < a.nnz;
         p0 += warps * kWarp) {
        const int64_t p = p0 + lane;
        int t = 0;
        int64_t src_row = -1;  // the host row to stage, or -1
        int64_t dst = -1;      // the rewritten index
        if (p < a.nnz) {
            if (p < bound[0] || p >= bound[a.T]) {
                flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
            } else {
                int lo = 0, hi = a.T - 1;  // the last table t with bound[t] <= p
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (bound[mid] <= p)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                t = lo;
                const int64_t r = static_cast<int64_t>(ind[p]);
                if (r >= 0 && r < a.num_rows[t]) {
                    const int32_t slot = a.slot_of[t][r];
                    if (slot >= 0) {
                        dst = slot;
                    } else {
                        const int m = atomicAdd(a.counters + t, 1);
                        if (m < a.stage_rows[t]) {
                            dst = a.cache_rows[t] + m;
                            src_row = r;
                        } else {
                            flag_status(a.status, DLRM_ERR_CAPACITY);  // no staging row left: pools as zero
                        }
                    }
                }  // else: out of range, stays -1
            }
            out[p] = static_cast<TI>(dst);
        }
        // the warp copies its missed rows, each by all lanes, kMissRows rows' loads in flight before the stores
        uint32_t miss = __ballot_sync(0xffffffffu, src_row >= 0);
        while (miss != 0) {
            const uint4* s[kMissRows];
            uint4* q[kMissRows];
#pragma unroll
            for (int u = 0; u < kMissRows; ++u) {
                s[u] = nullptr;
                q[u] = nullptr;
                if (miss != 0) {
                    const int l = __ffs(miss) - 1;
                    miss &= miss - 1;
                    const int tl = __shfl_sync(0xffffffffu, t, l);
                    const int64_t r = __shfl_sync(0xffffffffu, src_row, l);
                    const int64_t d = __shfl_sync(0xffffffffu, dst, l);
                    s[u] = reinterpret_cast<const uint4*>(static_cast<const char*>(a.host[tl]) + r * a.row_bytes);
                    q[u] = reinterpret_cast<uint4*>(static_cast<char*>(a.cache[tl]) + d * a.row_bytes);
                }
            }
            for (int c = lane; c < chunks; c += kWarp) {
                uint4 v[kMissRows];
#pragma unroll
                for (int u = 0; u < kMissRows; ++u)
                    if (s[u] != nullptr) v[u] = s[u][c];
#pragma unroll
                for (int u = 0; u < kMissRows; ++u)
                    if (q[u] != nullptr) q[u][c] = v[u];
            }
        }
    }
}

// Cache refill of one table: (1) the rows leaving the cache get slot -1; (2) rows[i] moves into slot i
// (copied from host memory) and slots past n hold nothing.
__global__ void __launch_bounds__(kTierThreads) uncache_kernel(int32_t* slot_of, const int64_t* slot_row, int64_t C,
                                                              int64_t V)
{
    for (int64_t s = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; s < C; s += int64_t{gridDim.x} * blockDim.x) {
        const int64_t r = slot_row[s];
        if (r >= 0 && r < V) slot_of[r] = -1;
    }
}

__global__ void __launch_bounds__(kTierThreads) fill_minus_one_kernel(int32_t* p32, int64_t n32, int64_t* p64, int64_t n64)
{
    const int64_t stride = int64_t{gridDim.x} * blockDim.x;
    for (int64_t i = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; i < n32; i += stride) p32[i] = -1;
    for (int64_t i = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; i < n64; i += stride) p64[i] = -1;
}

__global__ void __launch_bounds__(kTierThreads) fill_cache_kernel(const char* host, char* cache, int32_t* slot_of,
                                                                 int64_t* slot_row, const int64_t* rows, int64_t n,
                                                                 int64_t C, int64_t V, int row_bytes, int32_t* status)
{
    const int lane = threadIdx.x % kWarp;
    const int chunks = row_bytes / 16;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kTierThreads / kWarp);
    for (int64_t s = blockIdx.x * int64_t{kTierThreads / kWarp} + threadIdx.x / kWarp; s < C; s += warps) {
        const int64_t r = s < n ? rows[s] : -1;
        const bool ok = r >= 0 && r < V;
        if (s < n && !ok && lane == 0) flag_status(status, DLRM_ERR_INDEX_OOB);
        if (lane == 0) {
            slot_row[s] = ok ? r : -1;
            if (ok) slot_of[r] = static_cast<int32_t>(s);
        }
        if (ok) {
            const uint4* src = reinterpret_cast<const uint4*>(host + r * row_bytes);
            uint4* dst = reinterpret_cast<uint4*>(cache + s * row_bytes);
            for (int c = lane; c < chunks; c += kWarp) dst[c] = src[c];
        }
    }
}

}  // namespace

dlrm_status launch_tier_stage(const TierArgs& a, int index_type, void* out, cudaStream_t s)
{
    if (cudaMemsetAsync(a.counters, 0, sizeof(int32_t) * a.T, s) != cudaSuccess) return DLRM_ERR_CUDA;
    if (a.nnz == 0) return DLRM_OK;
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    const int64_t want = (a.nnz + kTierThreads - 1) / kTierThreads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    if (index_type == DLRM_I32)
        stage_kernel<int32_t><<<grid, kTierThreads, 0, s>>>(a, static_cast<int32_t*>(out));
    else
        stage_kernel<int64_t><<<grid, kTierThreads, 0, s>>>(a, static_cast<int64_t*>(out));
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

dlrm_status launch_tier_fill(const void* host, void* cache, int32_t* slot_of, int64_t* slot_row, const int64_t* rows,
                             int64_t n, int64_t C, int64_t V, int row_bytes, int32_t* status, cudaStream_t s)
{
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    if (C == 0) return DLRM_OK;
    const int64_t g1 = (C + kTierThreads - 1) / kTierThreads;
    uncache_kernel<<<static_cast<unsigned>(g1 < sms * 8 ? g1 : sms * 8), kTierThreads, 0, s>>>(slot_of, slot_row, C, V);
    const int64_t g2 = (C + kTierThreads / kWarp - 1) / (kTierThreads / kWarp);
    fill_cache_kernel<<<static_cast<unsigned>(g2 < sms * 8 ? g2 : sms * 8), kTierThreads, 0, s>>>(
        static_cast<const char*>(host), static_cast<char*>(cache), slot_of, slot_row, rows, n, C, V, row_bytes, status);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

dlrm_status launch_tier_init(int32_t* slot_of, int64_t V, int64_t* slot_row, int64_t C, cudaStream_t s)
{
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    fill_minus_one_kernel<<<static_cast<unsigned>(sms * 8), kTierThreads, 0, s>>>(slot_of, V, slot_row, C);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

}  // namespace dlrm
