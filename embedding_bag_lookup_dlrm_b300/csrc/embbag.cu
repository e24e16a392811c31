// embbag.cu -- the embedding-bag lookup on its own: pooled[b][t] = sum (or
// mean) of the rows of bag (t, b) ("DLRM", robocikowo.com, "Forward pass"
// step (2); bags of several IDs: "The embedding table is the model").
//
// HBM-bound gather.  A group of P lanes owns one bag, P = the row's 16-byte
// chunks (up to 32; D = 256 fp32 gives each lane two chunks), so a warp holds
// 32 / P bags.  The group reads the bag's offsets once, its indices P at a
// time with one load per lane, and then walks the lookups eight at a time:
// eight row loads in flight per lane before the adds.  Each sum is fp32 in
// lookup order, starting from its first term (so a one-lookup fp32 bag is a
// bit-exact copy of its row, -0.0 included); bf16 rows are widened exactly.
// An out-of-range index contributes nothing, still counts in a mean's L and
// is flagged; a bag whose every lookup is out of range, or an empty bag,
// pools to zero.  Bags are numbered table-major, as the offsets are, so
// consecutive groups read consecutive offsets and indices.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace dlrm {
namespace {

constexpr int kBagThreads = 256;
constexpr int kInFlight = 8;

template <int D, typename TE>
struct BagShape {
    static constexpr int kChunks = D * static_cast<int>(sizeof(TE)) / 16;  // 16-byte chunks per row
    static constexpr int P = kChunks < kWarp ? kChunks : kWarp;           // lanes per bag
    static constexpr int CPL = kChunks / P;                               // chunks per lane
    static constexpr int EPC = 16 / static_cast<int>(sizeof(TE));         // elements per chunk
    static constexpr int BPW = kWarp / P;                                 // bags per warp
};

template <typename TE>
__device__ __forceinline__ void widen_chunk(uint4 v, float (&f)[16 / sizeof(TE)])
{
    if constexpr (sizeof(TE) == 4) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    } else {
        bf16x8_to_f32(v, f);
    }
}

template <int D, typename TE, typename TI>
__global__ void __launch_bounds__(kBagThreads) embbag_kernel(const __grid_constant__ FwdArgs a)
{
    using S = BagShape<D, TE>;
    constexpr int P = S::P, CPL = S::CPL, EPC = S::EPC, BPW = S::BPW;
    const int lane = threadIdx.x % kWarp;
    const int grp = lane / P, gl = lane % P;                 // the group in the warp, the lane in the group
    const unsigned gmask = (P == kWarp) ? 0xffffffffu : (((1u << P) - 1u) << (grp * P));
    const int64_t nbags = static_cast<int64_t>(a.T) * a.B;
    const int64_t groups = static_cast<int64_t>(gridDim.x) * (kBagThreads / kWarp) * BPW;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int64_t first = static_cast<int64_t>(__ldg(static_cast<const TI*>(a.offsets)));
        const int64_t last = static_cast<int64_t>(__ldg(static_cast<const TI*>(a.offsets) + nbags));
        if (first != 0 || last != a.nnz) flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
    }
    const TI* off = static_cast<const TI*>(a.offsets);
    const TI* ind = static_cast<const TI*>(a.indices);
    const int64_t g0 = (static_cast<int64_t>(blockIdx.x) * (kBagThreads / kWarp) + threadIdx.x / kWarp) * BPW + grp;
    // every group of the warp runs the same number of iterations (shuffles stay warp-uniform)
    const int64_t warp_first = g0 - grp;
    for (int64_t w0 = warp_first; w0 < nbags; w0 += groups) {
        const int64_t bag = w0 + grp;
        const bool live = bag < nbags;
        const int t = live ? static_cast<int>(bag / a.B) : 0;
        const int64_t b = live ? bag - static_cast<int64_t>(t) * a.B : 0;
        int64_t s0 = 0, s1 = 0;
        if (live) {
            s0 = static_cast<int64_t>(__ldg(off + bag));
            s1 = static_cast<int64_t>(__ldg(off + bag + 1));
            if (s0 < 0 || s1 < s0 || s1 > a.nnz) {
                if (gl == 0) flag_status(a.status, DLRM_ERR_BAD_OFFSETS);  // treated as an empty bag
                s0 = s1 = 0;
            }
        }
        const int L = static_cast<int>(s1 - s0);
        const TE* table = live ? static_cast<const TE*>(a.tables[t]) : nullptr;
        const int64_t V = live ? a.num_rows[t] : 0;
        float acc[CPL][EPC];
        bool started = false;
        // the longest bag of the warp sets the trip count
        int Lmax = L;
#pragma unroll
        for (int o = P; o < kWarp; o <<= 1) Lmax = max(Lmax, __shfl_xor_sync(0xffffffffu, Lmax, o));
        for (int q0 = 0; q0 < Lmax; q0 += P) {
            int64_t my = -1;  // the index of lookup q0 + gl of this group's bag (-1: none or out of range)
            if (q0 + gl < L) {
                my = static_cast<int64_t>(__ldg(ind + s0 + q0 + gl));
                if (my < 0 || my >= V) {
                    flag_status(a.status, DLRM_ERR_INDEX_OOB);
                    my = -1;
                }
            }
            const int n = min(P, Lmax - q0);
            for (int u0 = 0; u0 < n; u0 += kInFlight) {
                uint4 raw[kInFlight][CPL];
                bool ok[kInFlight];
#pragma unroll
                for (int u = 0; u < kInFlight; ++u) {
                    const int src = grp * P + ((u0 + u) & (P - 1));
                    const int64_t r = __shfl_sync(0xffffffffu, my, src);
                    ok[u] = u0 + u < n && q0 + u0 + u < L && r >= 0;
                    if (ok[u]) {
                        const uint4* row = reinterpret_cast<const uint4*>(table + r * D);
#pragma unroll
                        for (int c = 0; c < CPL; ++c) raw[u][c] = __ldg(row + gl + c * P);
                    }
                }
#pragma unroll
                for (int u = 0; u < kInFlight; ++u) {
                    if (!ok[u]) continue;
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        float f[EPC];
                        widen_chunk<TE>(raw[u][c], f);
#pragma unroll
                        for (int e = 0; e < EPC; ++e) acc[c][e] = started ? acc[c][e] + f[e] : f[e];
                    }
                    started = true;
                }
            }
        }
        if (live) {
            float* dst = a.pooled_out + (b * a.T + t) * D;
            const float fl = static_cast<float>(L);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                float v[EPC];
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    float x = started ? acc[c][e] : 0.0f;
                    if (a.mean && started) x = __fdiv_rn(x, fl);
                    v[e] = x;
                }
                float4* d4 = reinterpret_cast<float4*>(dst + (gl + c * P) * EPC);
#pragma unroll
                for (int e = 0; e < EPC; e += 4) d4[e / 4] = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
            }
        }
        (void)gmask;
    }
}

template <int D, typename TE, typename TI>
dlrm_status launch_bags(const FwdArgs& a, cudaStream_t s)
{
    using S = BagShape<D, TE>;
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    const int64_t nbags = static_cast<int64_t>(a.T) * a.B;
    const int64_t per_block = (kBagThreads / kWarp) * S::BPW;
    const int64_t want = (nbags + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(sms) * 8 * 4;  // 8 blocks per SM, several waves of bags each
    embbag_kernel<D, TE, TI><<<static_cast<unsigned>(want < cap ? want : cap), kBagThreads, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

template <int D>
dlrm_status dispatch_bags(const FwdArgs& a, int dtype, int index_type, cudaStream_t s)
{
    if (dtype == DLRM_F32)
        return index_type == DLRM_I32 ? launch_bags<D, float, int32_t>(a, s) : launch_bags<D, float, int64_t>(a, s);
    return index_type == DLRM_I32 ? launch_bags<D, __nv_bfloat16, int32_t>(a, s)
                                  : launch_bags<D, __nv_bfloat16, int64_t>(a, s);
}

}  // namespace

dlrm_status launch_embbag(const FwdArgs& a, int dim, int dtype, int index_type, cudaStream_t s)
{
    switch (dim) {
        case 16: return dispatch_bags<16>(a, dtype, index_type, s);
        case 32: return dispatch_bags<32>(a, dtype, index_type, s);
        case 64: return dispatch_bags<64>(a, dtype, index_type, s);
        case 128: return dispatch_bags<128>(a, dtype, index_type, s);
        case 256: return dispatch_bags<256>(a, dtype, index_type, s);
        default: return DLRM_ERR_UNSUPPORTED;
    }
}

}  // namespace dlrm
