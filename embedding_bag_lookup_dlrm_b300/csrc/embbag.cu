// embbag.cu -- the embedding-bag lookup on its own: pooled[b][t] = sum (or
// mean) of the rows of bag (t, b) ("DLRM", robocikowo.com, "Forward pass"
// step (2); bags of several IDs: "The embedding table is the model").
//
// HBM-bound gather.  Rows of 128 bytes or more take the list form below.
// Narrower rows: a group of P lanes owns one bag, P = the row's 16-byte
// chunks, so a warp holds 32 / P bags.  The group reads the bag's offsets once, its indices P at a
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
#include "pool.cuh"

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

// The list form, for rows of at least 128 bytes.  A warp takes 32
// consecutive bags (lane l reads bag l's offsets, so the loads coalesce),
// flattens their lookups into one list, and walks it 32 lookups at a time:
// lane j resolves lookup j of the step (its bag by a 5-step search over the
// lanes' list ends, its index by one load, coalesced where the bags' ranges
// are contiguous) while the next step's indices are already on their way.
// The warp then streams the step's rows, a few at a time, each lane holding
// 1/32 of a row (16, 8 or 4 bytes; D = 256 fp32: two 16-byte pieces), adding
// each into the running bag's sum in lookup order; a finished bag is written
// once.  One-hot batches thus keep 32 bags' rows moving per warp instead of
// one.
//
// Rows in flight: kLaneBytesInFlight bytes per lane (4 rows of 512 bytes, 8 of
// 256), which keeps a thread within 64 registers, so that 4 CTAs of 8 warps
// share an SM.  Measured against 16 rows per warp at 2 CTAs per SM: the
// lookup of the training batch (bags of 1..8) 420 -> 273 us, one-hot rows of
// 512 bytes 297 -> 221 us, bf16 bags of 1..64 890 -> 649 us, rows of 256
// bytes 128 -> 94 us.  The warps, not the bytes each keeps moving, hide the
// latency of the lookups' dependent steps (offsets, index, row).
constexpr int kLaneBytesInFlight = 64;
constexpr int kListMinBlocks = 4;

template <int BYTES>
struct Piece;
template <>
struct Piece<16> {
    uint4 v;
    __device__ __forceinline__ void load(const void* p) { v = __ldg(static_cast<const uint4*>(p)); }
    __device__ __forceinline__ uint32_t w(int i) const { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
};
template <>
struct Piece<8> {
    uint2 v;
    __device__ __forceinline__ void load(const void* p) { v = __ldg(static_cast<const uint2*>(p)); }
    __device__ __forceinline__ uint32_t w(int i) const { return i == 0 ? v.x : v.y; }
};
template <>
struct Piece<4> {
    uint32_t v;
    __device__ __forceinline__ void load(const void* p) { v = __ldg(static_cast<const uint32_t*>(p)); }
    __device__ __forceinline__ uint32_t w(int) const { return v; }
};

template <int D, typename TE>
struct ListShape {
    static constexpr int kRowBytes = D * static_cast<int>(sizeof(TE));
    static constexpr int kLaneBytes = kRowBytes / kWarp;                 // 4 .. 32
    static constexpr int kPieceBytes = kLaneBytes > 16 ? 16 : kLaneBytes;
    static constexpr int kPieces = kLaneBytes / kPieceBytes;             // 1, or 2 (D = 256 fp32)
    static constexpr int kElems = kPieceBytes / static_cast<int>(sizeof(TE));  // elements per piece
};

template <int D, typename TE, typename TI>
__global__ void __launch_bounds__(kBagThreads, kListMinBlocks) embbag_list_kernel(const __grid_constant__ FwdArgs a)
{
    using S = ListShape<D, TE>;
    constexpr int NP = S::kPieces, NE = S::kElems, PB = S::kPieceBytes;
    constexpr int R = kLaneBytesInFlight / (NP * PB) > 0 ? kLaneBytesInFlight / (NP * PB) : 1;  // rows in flight
    using PieceT = Piece<PB>;
    const int lane = threadIdx.x % kWarp;
    const int64_t nbags = static_cast<int64_t>(a.T) * a.B;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kBagThreads / kWarp);
    const TI* off = static_cast<const TI*>(a.offsets);
    const TI* ind = static_cast<const TI*>(a.indices);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int64_t first = static_cast<int64_t>(__ldg(off));
        const int64_t last = static_cast<int64_t>(__ldg(off + nbags));
        if (first != 0 || last != a.nnz) flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
    }
    for (int64_t w0 = (blockIdx.x * int64_t{kBagThreads / kWarp} + threadIdx.x / kWarp) * kWarp; w0 < nbags;
         w0 += warps * kWarp) {
        // lane l: bag w0 + l
        const int64_t bag = w0 + lane;
        const bool live = bag < nbags;
        int64_t s0 = 0, s1 = 0;
        if (live) {
            s0 = static_cast<int64_t>(__ldg(off + bag));
            s1 = static_cast<int64_t>(__ldg(off + bag + 1));
            if (s0 < 0 || s1 < s0 || s1 > a.nnz) {
                flag_status(a.status, DLRM_ERR_BAD_OFFSETS);  // treated as an empty bag
                s0 = s1 = 0;
            }
        }
        const int len = static_cast<int>(s1 - s0);
        int incl = len;  // inclusive prefix of the bag lengths: the list end of each lane's bag
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
        const int t_lane = live ? static_cast<int>(bag / a.B) : 0;

        // lookup q of the list: its bag (lane) r and its index, or -1 when out of range
        auto resolve = [&](int q, int& r, int64_t& idx) {
            int at = 0;
#pragma unroll
            for (int bit = 16; bit > 0; bit >>= 1)
                if (__shfl_sync(0xffffffffu, incl, at + bit - 1) <= q) at += bit;
            r = at & (kWarp - 1);
            const int beg = __shfl_sync(0xffffffffu, incl - len, r);
            const int64_t st = __shfl_sync(0xffffffffu, s0, r);
            idx = q < total ? static_cast<int64_t>(__ldg(ind + st + (q - beg))) : -1;
        };

        // -0.0 is the additive identity that keeps every sum exact: -0.0 + x = x for every x, -0.0 included,
        // so a sum seeded with it equals the sum that starts from its first term
        float acc[NP][NE];
#pragma unroll
        for (int k = 0; k < NP; ++k)
#pragma unroll
            for (int e = 0; e < NE; ++e) acc[k][e] = -0.0f;
        int cur = -1;          // the bag (lane) being summed
        bool started = false;  // it has received a valid row
        auto finish = [&]() {  // write bag `cur` (all lanes)
            if (cur < 0) return;
            const int64_t bg = w0 + cur;
            const int t = static_cast<int>(bg / a.B);
            const int64_t b = bg - static_cast<int64_t>(t) * a.B;
            const int L = __shfl_sync(0xffffffffu, len, cur);
            float* dst = a.pooled_out + (b * a.T + t) * D;
#pragma unroll
            for (int k = 0; k < NP; ++k) {
                float v[NE];
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    float x = started ? acc[k][e] : 0.0f;
                    if (a.mean && started) x = __fdiv_rn(x, static_cast<float>(L));
                    v[e] = x;
                    acc[k][e] = -0.0f;  // seeded for the next bag
                }
                float* d = dst + (lane * NP + k) * NE;
                if constexpr (NE == 4) {
                    *reinterpret_cast<float4*>(d) = make_float4(v[0], v[1], v[2], v[3]);
                } else if constexpr (NE == 8) {
                    reinterpret_cast<float4*>(d)[0] = make_float4(v[0], v[1], v[2], v[3]);
                    reinterpret_cast<float4*>(d)[1] = make_float4(v[4], v[5], v[6], v[7]);
                } else if constexpr (NE == 2) {
                    *reinterpret_cast<float2*>(d) = make_float2(v[0], v[1]);
                } else {
                    d[0] = v[0];
                }
            }
        };
        // bags with no lookups never appear in the list: their zero rows first
        for (uint32_t empty = __ballot_sync(0xffffffffu, live && len == 0); empty != 0; empty &= empty - 1) {
            const int64_t bg = w0 + (__ffs(empty) - 1);
            const int t = static_cast<int>(bg / a.B);
            const int64_t b = bg - static_cast<int64_t>(t) * a.B;
            float* dst = a.pooled_out + (b * a.T + t) * D;
            for (int e = lane * 4; e < D; e += kWarp * 4)
                *reinterpret_cast<float4*>(dst + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        }

        int r_next = 0;
        int64_t i_next = -1;
        if (total > 0) resolve(lane, r_next, i_next);
        for (int q0 = 0; q0 < total; q0 += kWarp) {
            const int r_me = r_next;
            int64_t idx = i_next;
            if (q0 + kWarp < total) resolve(q0 + kWarp + lane, r_next, i_next);  // the next step's indices
            const int t_me = __shfl_sync(0xffffffffu, t_lane, r_me);
            const char* src = nullptr;
            if (q0 + lane < total) {
                if (idx >= 0 && idx < a.num_rows[t_me])
                    src = static_cast<const char*>(a.tables[t_me]) + static_cast<uint64_t>(idx) * S::kRowBytes;
                else
                    flag_status(a.status, DLRM_ERR_INDEX_OOB);  // contributes zero, still counts in L
            }
            const int tag = r_me | (src != nullptr ? 32 : 0);  // the lookup's bag and whether it has a row
            const int n = min(kWarp, total - q0);
#pragma unroll 1
            for (int h = 0; h < n; h += R) {
                PieceT raw[R][NP];
#pragma unroll
                for (int u = 0; u < R; ++u) {
                    const char* p = reinterpret_cast<const char*>(
                        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src), (h + u) & (kWarp - 1)));
                    if (h + u < n && p != nullptr) {
#pragma unroll
                        for (int k = 0; k < NP; ++k) raw[u][k].load(p + (lane * NP + k) * PB);
                    }
                }
#pragma unroll
                for (int u = 0; u < R; ++u) {
                    const int tu = __shfl_sync(0xffffffffu, tag, (h + u) & (kWarp - 1));
                    const int ru = tu & 31;
                    const bool valid = (tu & 32) != 0;
                    if (h + u >= n) continue;
                    if (ru != cur) {
                        finish();
                        cur = ru;
                        started = false;
                    }
                    if (!valid) continue;
#pragma unroll
                    for (int k = 0; k < NP; ++k) {
                        if constexpr (sizeof(TE) == 2) {  // mixed-precision adds, one per element
#pragma unroll
                            for (int e = 0; e < NE / 2; ++e) add_bf16_pair(acc[k][2 * e], acc[k][2 * e + 1], raw[u][k].w(e));
                        } else if constexpr (NE == 1) {
                            acc[k][0] += __uint_as_float(raw[u][k].w(0));
                        } else {
                            // packed adds (add.f32x2): each lane an ordinary fp32 add, rounded once
#pragma unroll
                            for (int e = 0; e < NE; e += 2) {
                                const float2 r2 = __fadd2_rn(make_float2(acc[k][e], acc[k][e + 1]),
                                                             make_float2(__uint_as_float(raw[u][k].w(e)),
                                                                         __uint_as_float(raw[u][k].w(e + 1))));
                                acc[k][e] = r2.x;
                                acc[k][e + 1] = r2.y;
                            }
                        }
                    }
                    started = true;
                }
            }
        }
        finish();
    }
}

template <int D, typename TE, typename TI>
dlrm_status launch_bags(const FwdArgs& a, cudaStream_t s)
{
    using S = BagShape<D, TE>;
    const int sms = sm_count();
    if (sms < 1) return DLRM_ERR_CUDA;
    if constexpr (D * sizeof(TE) >= 128) {
        const int64_t nbags = static_cast<int64_t>(a.T) * a.B;
        const int64_t want = (nbags + kBagThreads - 1) / kBagThreads;  // 32 bags per warp
        const int64_t cap = static_cast<int64_t>(sms) * 8;
        embbag_list_kernel<D, TE, TI><<<static_cast<unsigned>(want < cap ? want : cap), kBagThreads, 0, s>>>(a);
        return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
    }
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
