// fwd.cu -- sm_103a kernels of the DLRM sparse forward.
//
// One kernel template covers the fused forward and the interaction alone, for
// the shapes the tensor-core kernel (fwd_tc.cu) does not take:
//   kInteract  dot-product interaction    ("DLRM", robocikowo.com, "Forward pass" steps (3)-(4))
//   kFused     lookup + pooling (step (2); bags: "The embedding table is the model") and the
//              interaction, pooled vectors kept in shared memory
// (the lookup alone, kEmbbag, runs in embbag.cu).
//
// Work unit: one sample.  A "group" of G warps owns one sample at a time and
// stages its N = 1 + T vectors V (x first, then the pooled bags) as fp32 rows
// in shared memory:
//   * one-hot fp32 bags and the dense / pooled input rows are moved by the TMA
//     engine (cp.async.bulk, one instruction per row, completion counted on an
//     mbarrier), so a warp has every row of its sample in flight at once;
//   * multi-hot or bf16 bags are pooled in registers: each lane owns one or
//     more 16-byte chunks of a row, several rows per load instruction when a
//     row is narrower than a warp, up to 16 load instructions in flight per
//     warp (16 fp32 or 32 bf16 rows at D = 128), fp32 accumulation in lookup
//     order (packed fp32 adds, each rounded as a scalar add); when bags
//     average 8 or more lookups, two warps share a sample and take its bags
//     alternately;
//   * the strict upper triangle of V V^T is computed by register-blocked FFMA:
//     the rows are split into 4-row blocks with stride NB (block k = rows
//     k, k+NB, k+2NB, k+3NB) so that the lanes of a warp, each owning one
//     block pair, read consecutive rows from distinct shared-memory banks; a
//     lane accumulates a 4x4 tile of dot products over D;
//   * the triangle is staged in shared memory and the output row [x, triangle]
//     is written with coalesced stores.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "pool.cuh"

namespace dlrm {
namespace {

// Shared-memory layout of one group (byte offsets), shared by host and device.
struct GroupLayout {
    int T, N, NPAD, NB, K, S;  // S = fp32 row stride of V (D + 4)
    int off_start, off_len, off_V, off_tri, bytes;
};

__host__ __device__ inline GroupLayout make_layout(int T, int D, int mode)
{
    GroupLayout g;
    g.T = T;
    g.N = T + 1;
    g.NPAD = round_up(g.N, 4);
    g.NB = g.NPAD / 4;
    g.K = g.N * (g.N - 1) / 2;
    g.S = D + 4;
    int o = 16;                      // mbarrier
    g.off_start = o;                 // per row of V: int64 bag start, or TMA source address
    o += 8 * (T + 1);
    g.off_len = o;                   // per row of V: bag length, or -1 when the TMA engine moves it
    o = round_up(o + 4 * (T + 1), 16);
    g.off_V = o;
    o += 4 * g.NPAD * g.S;
    g.off_tri = o;
    if (mode != kEmbbag) o += 4 * g.K;
    g.bytes = round_up(o, 128);
    return g;
}

template <int G>
__device__ __forceinline__ void group_sync()
{
    if (G == 1)
        __syncwarp();
    else
        __syncthreads();  // G > 1 runs one group per CTA
}

template <typename TI>
__device__ __forceinline__ int64_t load_index(const void* p, int64_t i)
{
    return static_cast<int64_t>(__ldg(static_cast<const TI*>(p) + i));
}

// ---------------------------------------------------------------------------
// Pool one bag in registers into an fp32 shared-memory row (one warp), up to
// MAXU row-load instructions in flight.
// ---------------------------------------------------------------------------
template <int D, typename TE, typename TI, int MAXU = 16>
__device__ void pool_bag_warp(const TE* __restrict__ table, int64_t V_t, const void* indices, int64_t start,
                              int L, bool mean, float* vrow, int lane, int32_t* status)
{
    constexpr int EPC = 16 / sizeof(TE);         // elements per 16-byte chunk
    constexpr int CPR = D / EPC;                 // chunks per row
    constexpr int LPR = CPR < kWarp ? CPR : kWarp;  // lanes per row
    constexpr int CPL = CPR / LPR;               // chunks per lane
    constexpr int RPI = kWarp / LPR;             // rows per load instruction
    constexpr int U0 = (kWarp / RPI) < MAXU ? (kWarp / RPI) : MAXU;
    constexpr int U = (U0 / CPL) > 0 ? (U0 / CPL) : 1;  // load instructions in flight
    constexpr int STEP = RPI * U;                // lookups per step (divides 32)
    static_assert(kWarp % STEP == 0, "step must divide the warp");

    const int h = lane / LPR;   // which of the RPI rows this lane loads
    const int c0 = lane % LPR;  // first chunk of the row this lane owns

    float acc[CPL][EPC];
#pragma unroll
    for (int k = 0; k < CPL; ++k)
#pragma unroll
        for (int e = 0; e < EPC; ++e) acc[k][e] = -0.0f;  // additive identity that keeps -0.0

    bool any_valid = false;
    for (int qb = 0; qb < L; qb += kWarp) {
        const int nq = min(kWarp, L - qb);
        const int64_t my_idx = lane < nq ? load_index<TI>(indices, start + qb + lane) : 0;
        for (int qq = 0; qq < nq; qq += STEP) {
            uint4 raw[U][CPL];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = qq + h + RPI * u;
                const int64_t r = __shfl_sync(0xffffffffu, my_idx, q & (kWarp - 1));
                const bool in_bag = q < nq;
                ok[u] = in_bag && r >= 0 && r < V_t;
                if (in_bag && !ok[u] && c0 == 0) flag_status(status, DLRM_ERR_INDEX_OOB);
                if (ok[u]) {
                    const TE* row = table + r * D;
#pragma unroll
                    for (int k = 0; k < CPL; ++k)
                        raw[u][k] = __ldg(reinterpret_cast<const uint4*>(row + (c0 + k * LPR) * EPC));
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!ok[u]) continue;
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    if constexpr (sizeof(TE) == 2) {
                        // mixed-precision adds (add.f32.bf16): the bf16 element, widened exactly, plus the fp32
                        // sum, rounded once; the same result as widening first, in one instruction per element
                        const uint32_t w[4] = {raw[u][k].x, raw[u][k].y, raw[u][k].z, raw[u][k].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) add_bf16_pair(acc[k][2 * e], acc[k][2 * e + 1], w[e]);
                    } else {
                        // packed adds (add.f32x2): each lane an ordinary fp32 add, rounded once
                        const float2 s0 = __fadd2_rn(make_float2(acc[k][0], acc[k][1]),
                                                     make_float2(__uint_as_float(raw[u][k].x), __uint_as_float(raw[u][k].y)));
                        const float2 s1 = __fadd2_rn(make_float2(acc[k][2], acc[k][3]),
                                                     make_float2(__uint_as_float(raw[u][k].z), __uint_as_float(raw[u][k].w)));
                        acc[k][0] = s0.x;
                        acc[k][1] = s0.y;
                        acc[k][2] = s1.x;
                        acc[k][3] = s1.y;
                    }
                }
            }
            any_valid |= __any_sync(0xffffffffu, ok[0]) != 0;
#pragma unroll
            for (int u = 1; u < U; ++u) any_valid |= __any_sync(0xffffffffu, ok[u]) != 0;
        }
    }
    // Fold the RPI interleaved partial sums (fixed order: reproducible).
#pragma unroll
    for (int s = LPR; s < kWarp; s <<= 1)
#pragma unroll
        for (int k = 0; k < CPL; ++k)
#pragma unroll
            for (int e = 0; e < EPC; ++e) acc[k][e] += __shfl_xor_sync(0xffffffffu, acc[k][e], s);

    if (h == 0) {
        const float len_f = static_cast<float>(L);
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            float v[EPC];
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                float a = any_valid ? acc[k][e] : 0.0f;
                if (mean && any_valid) a = __fdiv_rn(a, len_f);
                v[e] = a;
            }
            float* dst = vrow + (c0 + k * LPR) * EPC;
#pragma unroll
            for (int e = 0; e < EPC; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
    }
}

// ---------------------------------------------------------------------------
// Strict upper triangle of V V^T into tri[] (group-cooperative).
// ---------------------------------------------------------------------------
template <int D>
__device__ void gram_upper(const float* __restrict__ V, const GroupLayout& g, float* __restrict__ tri, int gl,
                           int GT)
{
    const int NB = g.NB, N = g.N, S = g.S;
    const int NBP = NB * (NB + 1) / 2;
    for (int bp = gl; bp < NBP; bp += GT) {
        int bi = 0, rem = bp;
        while (rem >= NB - bi) {
            rem -= NB - bi;
            ++bi;
        }
        const int bj = bi + rem;
        const float* ri[4];
        const float* rj[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            ri[r] = V + (bi + NB * r) * S;
            rj[r] = V + (bj + NB * r) * S;
        }
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int s = 0; s < 4; ++s) acc[r][s] = 0.0f;

#pragma unroll 4
        for (int c = 0; c < D; c += 4) {
            float4 a[4], b[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4*>(ri[r] + c);
#pragma unroll
            for (int s = 0; s < 4; ++s) b[s] = *reinterpret_cast<const float4*>(rj[s] + c);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    float t = acc[r][s];
                    t = fmaf(a[r].x, b[s].x, t);
                    t = fmaf(a[r].y, b[s].y, t);
                    t = fmaf(a[r].z, b[s].z, t);
                    t = fmaf(a[r].w, b[s].w, t);
                    acc[r][s] = t;
                }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int i = bi + NB * r, j = bj + NB * s;
                const bool keep = (bi != bj) ? true : (r < s);
                if (keep && i < N && j < N) {
                    const int lo = i < j ? i : j, hi = i < j ? j : i;
                    tri[tri_index(lo, hi, N)] = acc[r][s];
                }
            }
    }
}

// ---------------------------------------------------------------------------
// The forward kernel.
// ---------------------------------------------------------------------------
// Samples of long bags (G = 2 warps each) keep 8 row loads in flight per warp within 85 registers, so that
// 12 of their CTAs (of 64 threads) share an SM instead of 8: workload 3 (bf16 bags of 1..64) 743.5 -> 616.7 us
// against 16 loads in flight per warp.  More warps, not more loads per warp, hide the lookups' latency.
template <int G>
constexpr int ffma_min_blocks() { return G == 2 ? 3 : 1; }
template <int G>
constexpr int ffma_loads_in_flight() { return G == 2 ? 8 : 16; }

template <int D, typename TE, typename TI, int MODE, int G>
__global__ void __launch_bounds__(256, ffma_min_blocks<G>()) forward_kernel(const __grid_constant__ FwdArgs a,
                                                                           int groups_per_cta)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int GT = G * kWarp;
    const GroupLayout g = make_layout(a.T, D, MODE);
    const int group = threadIdx.x / GT;
    const int gl = threadIdx.x % GT;
    const int lane = gl % kWarp;
    const int wig = gl / kWarp;  // warp within group
    const int64_t b = static_cast<int64_t>(blockIdx.x) * groups_per_cta + group;

    if (blockIdx.x == 0 && threadIdx.x == 0 && MODE != kInteract) {
        const int64_t first = load_index<TI>(a.offsets, 0);
        const int64_t last = load_index<TI>(a.offsets, static_cast<int64_t>(a.T) * a.B);
        if (first != 0 || last != a.nnz) flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
    }
    if (b >= a.B) return;  // whole group leaves together (G > 1 has one group per CTA)

    unsigned char* base = smem + group * g.bytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(base);
    int64_t* slot = reinterpret_cast<int64_t*>(base + g.off_start);
    int* lens = reinterpret_cast<int*>(base + g.off_len);
    float* V = reinterpret_cast<float*>(base + g.off_V);
    float* tri = reinterpret_cast<float*>(base + g.off_tri);
    const int T = a.T, S = g.S;
    constexpr uint32_t kRowBytes = D * 4;

    if (gl == 0) {
        mbar_init(bar, GT);
        fence_mbar_init();
    }
    group_sync<G>();

    // ---- pass 1: metadata; rows the TMA engine can move unchanged ----
    // Row k of V: 0 = dense x, 1 + t = bag t.  slot[k] holds the bag start
    // (pooled in registers) or the global address of a row to copy.
    uint32_t my_bytes = 0;
    for (int k = gl; k <= T; k += GT) {
        int len = -1;
        int64_t sv = 0;
        if (k == 0) {
            if (MODE != kEmbbag) {
                sv = reinterpret_cast<int64_t>(a.dense + b * D);
                my_bytes += kRowBytes;
            } else {
                len = 0;  // unused row
            }
        } else if (MODE == kInteract) {
            sv = reinterpret_cast<int64_t>(a.pooled_in + (b * T + (k - 1)) * D);
            my_bytes += kRowBytes;
        } else {
            const int t = k - 1;
            const int64_t bag = static_cast<int64_t>(t) * a.B + b;
            const int64_t s0 = load_index<TI>(a.offsets, bag);
            const int64_t s1 = load_index<TI>(a.offsets, bag + 1);
            len = 0;
            if (s0 < 0 || s1 < s0 || s1 > a.nnz)
                flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
            else
                len = static_cast<int>(s1 - s0);
            sv = s0;
            if (sizeof(TE) == 4 && len == 1) {
                const int64_t r = load_index<TI>(a.indices, s0);
                if (r >= 0 && r < a.num_rows[t]) {
                    sv = reinterpret_cast<int64_t>(static_cast<const float*>(a.tables[t]) + r * D);
                    my_bytes += kRowBytes;
                    len = -1;
                } else {
                    flag_status(a.status, DLRM_ERR_INDEX_OOB);
                    len = 0;  // contributes nothing: pooled as an empty bag
                }
            }
        }
        slot[k] = sv;
        lens[k] = len;
    }
    if (my_bytes > 0)
        mbar_arrive_expect_tx(bar, my_bytes);
    else
        mbar_arrive(bar);
    for (int k = gl; k <= T; k += GT)
        if (lens[k] < 0) bulk_g2s(V + k * S, reinterpret_cast<const void*>(slot[k]), kRowBytes, bar);

    // zero the padding rows of V so their dot products vanish
    if (MODE != kEmbbag) {
        for (int e = gl * 4; e < (g.NPAD - g.N) * S; e += GT * 4)
            *reinterpret_cast<float4*>(V + g.N * S + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    group_sync<G>();

    // ---- pass 2: bags pooled in registers (multi-hot, bf16, empty) ----
    if (MODE != kInteract) {
        for (int t = wig; t < T; t += G) {
            const int len = lens[t + 1];
            if (len < 0) continue;
            pool_bag_warp<D, TE, TI, ffma_loads_in_flight<G>()>(static_cast<const TE*>(a.tables[t]), a.num_rows[t],
                                                                a.indices, slot[t + 1],
                                     len, a.mean != 0, V + (t + 1) * S, lane, a.status);
        }
    }

    // ---- wait for the TMA rows (bounded; the whole group agrees) ----
    const bool landed = mbar_wait_bounded(bar, 0);
    const bool failed = (G == 1) ? (__any_sync(0xffffffffu, !landed) != 0) : (__syncthreads_or(!landed) != 0);
    if (failed) {
        if (gl == 0) flag_status(a.status, DLRM_ERR_TIMEOUT);
        return;
    }
    if (G == 1) __syncwarp();

    // ---- pooled vectors out (embbag, or fused with pooled_save) ----
    if (MODE == kEmbbag || (MODE == kFused && a.pooled_out != nullptr)) {
        float* p = a.pooled_out + b * T * D;
        for (int e = gl * 4; e < T * D; e += GT * 4) {
            const int t = e / D, d = e - t * D;
            *reinterpret_cast<float4*>(p + e) = *reinterpret_cast<const float4*>(V + (t + 1) * S + d);
        }
    }
    if (MODE == kEmbbag) return;

    // ---- interaction: strict upper triangle of the Gram matrix ----
    gram_upper<D>(V, g, tri, gl, GT);
    group_sync<G>();

    // ---- out[b] = [x, triangle] ----
    const int W = D + g.K;
    float* o = a.out + b * W;
    for (int k = gl; k < W; k += GT) o[k] = (k < D) ? V[k] : tri[k - D];
}

// ---------------------------------------------------------------------------
// Host side: configuration and dispatch.
// ---------------------------------------------------------------------------
constexpr int kMaxSmem = 227 * 1024;

template <int D, typename TE, typename TI, int MODE, int G>
dlrm_status launch_one(const FwdArgs& a, cudaStream_t stream)
{
    const GroupLayout g = make_layout(a.T, D, MODE);
    int groups = 1;
    if (G == 1) {
        groups = kMaxSmem / g.bytes;
        if (groups > 4) groups = 4;
        if (groups < 1) return DLRM_ERR_UNSUPPORTED;
    } else if (g.bytes > kMaxSmem) {
        return DLRM_ERR_UNSUPPORTED;
    }
    const size_t smem = static_cast<size_t>(groups) * g.bytes;
    auto kern = forward_kernel<D, TE, TI, MODE, G>;
    // set on every launch: the attribute belongs to the current device's context
    if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) !=
                                cudaSuccess)
        return DLRM_ERR_CUDA;
    const int64_t blocks = (a.B + groups - 1) / groups;
    if (blocks > 0x7fffffff) return DLRM_ERR_UNSUPPORTED;
    kern<<<static_cast<unsigned>(blocks), groups * G * kWarp, smem, stream>>>(a, groups);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

// A sample's triangle is shared by 8 warps once it has many 4x4 block pairs.
inline bool wide_interaction(int T)
{
    const int NB = round_up(T + 1, 4) / 4;
    return NB * (NB + 1) / 2 > 64;
}

// Bags of 8 or more lookups on average: two warps pool a sample's bags, so a
// sample's shared memory keeps twice the row loads in flight.
inline bool long_bags(const FwdArgs& a) { return a.nnz >= 8 * static_cast<int64_t>(a.T) * a.B; }

template <int D, typename TE, typename TI>
dlrm_status dispatch_mode(int mode, const FwdArgs& a, cudaStream_t s)
{
    const bool wide = wide_interaction(a.T);
    switch (mode) {
        case kFused:
            if (wide) return launch_one<D, TE, TI, kFused, 8>(a, s);
            return long_bags(a) ? launch_one<D, TE, TI, kFused, 2>(a, s) : launch_one<D, TE, TI, kFused, 1>(a, s);
        default: return DLRM_ERR_UNSUPPORTED;
    }
}

template <int D>
dlrm_status dispatch_types(int mode, const FwdArgs& a, int dtype, int index_type, cudaStream_t s)
{
    if (mode == kInteract)
        return wide_interaction(a.T) ? launch_one<D, float, int32_t, kInteract, 8>(a, s)
                                     : launch_one<D, float, int32_t, kInteract, 1>(a, s);
    if (dtype == DLRM_F32)
        return index_type == DLRM_I32 ? dispatch_mode<D, float, int32_t>(mode, a, s)
                                      : dispatch_mode<D, float, int64_t>(mode, a, s);
    return index_type == DLRM_I32 ? dispatch_mode<D, __nv_bfloat16, int32_t>(mode, a, s)
                                  : dispatch_mode<D, __nv_bfloat16, int64_t>(mode, a, s);
}

}  // namespace

dlrm_status launch_forward(int mode, const FwdArgs& a, int dim, int dtype, int index_type, cudaStream_t s)
{
    if (mode == kEmbbag) return launch_embbag(a, dim, dtype, index_type, s);
    // Training forward of bags averaging more than 1.25 lookups: the pooled vectors are written for the
    // backward anyway, so the lookup kernel pools them at its own pace and the tensor-core interaction
    // reads them back.  Re-reading B*T*D*4 bytes costs less than the fused kernel's gather, split and
    // MMA phases waiting on each other inside a CTA (on bags of 1..8: 540 against 588 us per batch of
    // 32,768).  The sums are the same: each bag in lookup order, in fp32.
    if (mode == kFused && a.pooled_out != nullptr && forward_tc_supported(mode, dim, a.T, a.B, a.nnz) &&
        4 * a.nnz > 5 * static_cast<int64_t>(a.T) * a.B) {
        const dlrm_status st = launch_embbag(a, dim, dtype, index_type, s);
        if (st != DLRM_OK) return st;
        FwdArgs b = a;
        b.pooled_in = a.pooled_out;
        return launch_forward_tc(kInteract, b, dim, DLRM_F32, DLRM_I32, s);
    }
    if (forward_tc_supported(mode, dim, a.T, a.B, a.nnz)) return launch_forward_tc(mode, a, dim, dtype, index_type, s);
    switch (dim) {
        case 16: return dispatch_types<16>(mode, a, dtype, index_type, s);
        case 32: return dispatch_types<32>(mode, a, dtype, index_type, s);
        case 64: return dispatch_types<64>(mode, a, dtype, index_type, s);
        case 128: return dispatch_types<128>(mode, a, dtype, index_type, s);
        case 256: return dispatch_types<256>(mode, a, dtype, index_type, s);
        default: return DLRM_ERR_UNSUPPORTED;
    }
}

}  // namespace dlrm
