// hash.cu -- the raw-ID hashing pre-pass: raw 64-bit feature IDs to rows of
// their tables, rows[p] = raw[p] mod V_t (the ID unsigned), t the table whose
// bags hold lookup p.  Hashing IDs into tables of fixed size is the systems
// choice "Deep Learning Recommendation Model (DLRM)" (notes.helloworld.co.in),
// "Why it is mostly a systems problem" names; the modulo is its plainest form.
//
// One pass over the lookups, HBM-bound: 8 bytes read and 4 (int32) or 8
// (int64) written per lookup.  The table of a lookup comes from a binary
// search over the T + 1 table boundaries offsets[t*B], staged in shared
// memory; the 64-bit remainder from a multiply-high by a per-table
// reciprocal: with m = floor((2^64 - 1) / V), q = floor(x m / 2^64) lies in
// [floor(x / V) - 2, floor(x / V)], so r = x - q V < 3V needs at most two
// subtractions of V.
#include "common.cuh"
#include "internal.h"

namespace dlrm {
namespace {

constexpr int kHashThreads = 256;

__device__ __forceinline__ uint64_t mod_u64(uint64_t x, uint64_t V, uint64_t m)
{
    const uint64_t q = __umul64hi(x, m);
    uint64_t r = x - q * V;
    if (r >= V) r -= V;
    if (r >= V) r -= V;
    return r;
}

template <typename TI>
__global__ void __launch_bounds__(kHashThreads) hash_kernel(const __grid_constant__ HashArgs a)
{
    __shared__ int64_t bound[DLRM_MAX_TABLES + 1];
    const TI* off = static_cast<const TI*>(a.offsets);
    for (int t = threadIdx.x; t <= a.T; t += blockDim.x) bound[t] = static_cast<int64_t>(off[static_cast<int64_t>(t) * a.B]);
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        bool bad = bound[0] != 0 || bound[a.T] != a.nnz;
        for (int t = 0; t < a.T; ++t) bad |= bound[t + 1] < bound[t];
        if (bad) flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
    }
    TI* rows = static_cast<TI*>(a.rows);
    for (int64_t p = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; p < a.nnz; p += int64_t{gridDim.x} * blockDim.x) {
        const uint64_t x = a.raw[p];
        if (p < bound[0] || p >= bound[a.T]) {  // in no table's range: malformed offsets
            flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
            rows[p] = 0;
            continue;
        }
        int lo = 0, hi = a.T - 1;  // the last table t with bound[t] <= p
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (bound[mid] <= p)
                lo = mid;
            else
                hi = mid - 1;
        }
        rows[p] = static_cast<TI>(mod_u64(x, a.num_rows[lo], a.magic[lo]));
    }
}

}  // namespace

dlrm_status launch_hash(const HashArgs& a, int index_type, cudaStream_t s)
{
    if (a.nnz == 0) return DLRM_OK;
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    const int64_t want = (a.nnz + kHashThreads - 1) / kHashThreads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    if (index_type == DLRM_I32)
        hash_kernel<int32_t><<<grid, kHashThreads, 0, s>>>(a);
    else
        hash_kernel<int64_t><<<grid, kHashThreads, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

}  // namespace dlrm
