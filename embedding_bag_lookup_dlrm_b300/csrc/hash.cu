// hash.cu -- the raw-ID hashing pre-pass: raw 64-bit feature IDs to rows of
// their tables, rows[p] = raw[p] mod V_t (the ID unsigned), t the table whose
// bags hold lookup p.  Hashing IDs into tables of fixed size is the systems
// choice "Deep Learning Recommendation Model (DLRM)" (notes.helloworld.co.in),
// "Why it is mostly a systems problem" names; the modulo is its plainest form.
//
// One pass over the lookups, HBM-bound: 8 bytes read and 4 (int32) or 8
// (int64) written per lookup, four lookups per thread in 16-byte vectors when
// both buffers allow it.  The table of a lookup comes from a binary search over
// the T + 1 table boundaries offsets[t*B], staged in shared memory (a thread's
// next lookups usually stay in the same table and skip the search); the 64-bit remainder from a multiply-high by a per-table
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

// The table of position p: the last t with bound[t] <= p (bound[0] <= p < bound[T]).
__device__ __forceinline__ int table_of(const int64_t* bound, int T, int64_t p)
{
    int lo = 0, hi = T - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (bound[mid] <= p)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// One lookup; returns its row (0 and a flag when p is in no table's range).
__device__ __forceinline__ uint64_t hash_one(const HashArgs& a, const int64_t* bound, int& t, int64_t p, uint64_t x)
{
    if (p < bound[0] || p >= bound[a.T]) {
        flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
        return 0;
    }
    if (p >= bound[t + 1] || p < bound[t]) t = table_of(bound, a.T, p);  // past the table of the lookup before
    return mod_u64(x, a.num_rows[t], a.magic[t]);
}

// VEC: 4 consecutive lookups per thread, IDs in two 16-byte loads, rows in one
// (int32) or two (int64) 16-byte stores; both buffers 16-byte aligned.
template <typename TI, bool VEC>
__global__ void __launch_bounds__(kHashThreads) hash_kernel(const __grid_constant__ HashArgs a)
{
    __shared__ int64_t bound[DLRM_MAX_TABLES + 2];
    const TI* off = static_cast<const TI*>(a.offsets);
    for (int t = threadIdx.x; t <= a.T; t += blockDim.x) bound[t] = static_cast<int64_t>(off[static_cast<int64_t>(t) * a.B]);
    if (threadIdx.x == 0) bound[a.T + 1] = INT64_MAX;  // so that bound[t + 1] exists for t = T
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        bool bad = bound[0] != 0 || bound[a.T] != a.nnz;
        for (int t = 0; t < a.T; ++t) bad |= bound[t + 1] < bound[t];
        if (bad) flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
    }
    TI* rows = static_cast<TI*>(a.rows);
    const int64_t stride = int64_t{gridDim.x} * blockDim.x;
    int t = 0;
    if (VEC) {
        const int64_t n4 = a.nnz / 4;
        for (int64_t q = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; q < n4; q += stride) {
            const ulonglong2 x01 = reinterpret_cast<const ulonglong2*>(a.raw)[2 * q];
            const ulonglong2 x23 = reinterpret_cast<const ulonglong2*>(a.raw)[2 * q + 1];
            const int64_t p = 4 * q;
            if (p >= bound[0] && p < bound[a.T]) t = table_of(bound, a.T, p);
            const uint64_t r0 = hash_one(a, bound, t, p, x01.x), r1 = hash_one(a, bound, t, p + 1, x01.y);
            const uint64_t r2 = hash_one(a, bound, t, p + 2, x23.x), r3 = hash_one(a, bound, t, p + 3, x23.y);
            if constexpr (sizeof(TI) == 4) {
                reinterpret_cast<int4*>(rows)[q] = make_int4(static_cast<int>(r0), static_cast<int>(r1),
                                                             static_cast<int>(r2), static_cast<int>(r3));
            } else {
                reinterpret_cast<longlong2*>(rows)[2 * q] = make_longlong2(static_cast<long long>(r0),
                                                                           static_cast<long long>(r1));
                reinterpret_cast<longlong2*>(rows)[2 * q + 1] = make_longlong2(static_cast<long long>(r2),
                                                                               static_cast<long long>(r3));
            }
        }
    }
    const int64_t first = VEC ? a.nnz / 4 * 4 : 0;  // the ragged tail (or everything) one lookup per thread
    for (int64_t p = first + blockIdx.x * int64_t{blockDim.x} + threadIdx.x; p < a.nnz; p += stride)
        rows[p] = static_cast<TI>(hash_one(a, bound, t, p, a.raw[p]));
}

}  // namespace

dlrm_status launch_hash(const HashArgs& a, int index_type, cudaStream_t s)
{
    if (a.nnz == 0) return DLRM_OK;
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    const bool vec = ((reinterpret_cast<uintptr_t>(a.raw) | reinterpret_cast<uintptr_t>(a.rows)) & 15u) == 0;
    const int64_t per_thread = vec ? 4 : 1;
    const int64_t want = (a.nnz / per_thread + kHashThreads - 1) / kHashThreads + 1;
    const int64_t cap = static_cast<int64_t>(sms) * 16;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    if (index_type == DLRM_I32) {
        if (vec)
            hash_kernel<int32_t, true><<<grid, kHashThreads, 0, s>>>(a);
        else
            hash_kernel<int32_t, false><<<grid, kHashThreads, 0, s>>>(a);
    } else {
        if (vec)
            hash_kernel<int64_t, true><<<grid, kHashThreads, 0, s>>>(a);
        else
            hash_kernel<int64_t, false><<<grid, kHashThreads, 0, s>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

}  // namespace dlrm
