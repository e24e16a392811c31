// bwd.cu -- sm_103a kernels of the DLRM sparse training step:
//   interaction backward -> lookup keys -> stable LSD radix sort by row ->
//   ordered segment sums -> row-wise Adagrad, in place.
//
// Training with Adagrad: "DLRM" (robocikowo.com), "Forward pass", last
// sentence.  The backward of out = [x, triu(V V^T)] is calculus on steps
// (3)-(4) of the same paragraph:  dV_i = sum_{j != i} g(i,j) V_j with
// g(i,j) = g(j,i) the upstream gradient of pair (i,j).
//
// Reproducibility: every floating-point sum here runs in an order fixed by
// the data layout alone (the stable sort keeps lookups of a row in lookup
// order; long runs are cut into fixed-size chunks whose partial sums are
// added in chunk order), so two calls on the same inputs give the same bits.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace dlrm {
namespace {

constexpr uint32_t kSentinel = 0xFFFFFFFFu;  // key of a lookup that updates nothing

// ---- workspace layout ------------------------------------------------------
constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;
constexpr int kSortTile = kSortThreads * kSortItems;  // 4096 keys per tile
constexpr int kMaxRadixBits = 9;  // digit width of a pass: up to 9 bits
constexpr int kMaxBins = 1 << kMaxRadixBits;
constexpr int kChunk = 128;  // sorted lookups per segment-reduction warp
constexpr int kSegThreads = 128;

inline size_t align256(size_t x) { return (x + 255) & ~size_t{255}; }

struct Workspace {
    float* dP;          // B x T x D
    uint32_t* keys[2];  // nnz each, ping-pong
    uint32_t* vals[2];
    uint32_t* counts;   // kMaxBins x num_tiles
    uint32_t* bin_total;  // kMaxBins
    float* partial;     // 2 x num_chunks x D
    int64_t num_tiles, num_chunks;
};

// with_dP: the workspace holds dP (the training step, or a scaled copy of a given pooled gradient).
Workspace carve(void* base, int64_t B, int32_t T, int32_t D, int64_t nnz, bool with_dP, size_t* total)
{
    Workspace w{};
    w.num_tiles = (nnz + kSortTile - 1) / kSortTile;
    w.num_chunks = (nnz + kChunk - 1) / kChunk;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    const size_t o_dP = with_dP ? take(sizeof(float) * B * T * D) : 0;
    size_t o_k[2], o_v[2];
    for (int i = 0; i < 2; ++i) {
        o_k[i] = take(sizeof(uint32_t) * nnz);
        o_v[i] = take(sizeof(uint32_t) * nnz);
    }
    const size_t o_cnt = take(sizeof(uint32_t) * kMaxBins * (w.num_tiles > 0 ? w.num_tiles : 1));
    const size_t o_tot = take(sizeof(uint32_t) * kMaxBins);
    const size_t o_par = take(sizeof(float) * 2 * (w.num_chunks > 0 ? w.num_chunks : 1) * D);
    if (total) *total = o;
    if (base) {
        char* p = static_cast<char*>(base);
        w.dP = with_dP ? reinterpret_cast<float*>(p + o_dP) : nullptr;
        for (int i = 0; i < 2; ++i) {
            w.keys[i] = reinterpret_cast<uint32_t*>(p + o_k[i]);
            w.vals[i] = reinterpret_cast<uint32_t*>(p + o_v[i]);
        }
        w.counts = reinterpret_cast<uint32_t*>(p + o_cnt);
        w.bin_total = reinterpret_cast<uint32_t*>(p + o_tot);
        w.partial = reinterpret_cast<float*>(p + o_par);
    }
    return w;
}

template <typename TI>
__device__ __forceinline__ int64_t ld_index(const void* p, int64_t i)
{
    return static_cast<int64_t>(__ldg(static_cast<const TI*>(p) + i));
}

// ---------------------------------------------------------------------------
// 1. Interaction backward.  One group of G warps per sample.  V (x, then the
// pooled rows) arrives by two bulk copies; the symmetric upstream matrix g
// (zero diagonal) is built in shared memory from the triangle.  Each lane owns
// 16-byte column chunks of V and accumulates an 8-row block of dV = g V,
// summing over j in increasing order, with packed fp32 FMAs (fma.rn.f32x2:
// two independent fused multiply-adds, each rounded once, as fmaf) on pairs of
// rows: one broadcast 16-byte load of g gives the factors of four rows, and
// each V value is paired with itself in registers.  Shared-memory bandwidth
// bounds this kernel, so g is kept once and the pairing is done in registers.
// ---------------------------------------------------------------------------
struct BwdLayout {
    int N, NP, K, W;  // NP = N rounded up to 8 (rows of g); W = D + K (upstream row)
    int off_V, off_g, off_go, bytes;
};

__host__ __device__ inline BwdLayout make_bwd_layout(int T, int D)
{
    BwdLayout l;
    l.N = T + 1;
    l.NP = round_up(l.N, 8);
    l.K = l.N * (l.N - 1) / 2;
    l.W = D + l.K;
    int o = 16;  // mbarrier
    l.off_V = o;
    o += 4 * l.N * D;
    l.off_g = o;
    o += 4 * l.NP * l.NP;
    l.off_go = o;
    o += 4 * l.W;
    l.bytes = round_up(o, 128);
    return l;
}

// NQ row pairs of a block of dV at one lane's 4 columns, summed over j in
// increasing order: p[q][c] += (g(i0+2q, j), g(i0+2q+1, j)) * V[j][col+c],
// with v pointing at V[0][col] and g at column i0 of row 0 of g.
template <int NQ>
__device__ __forceinline__ void grad_rows(const float* v, const float* g, int N, int NP, int D, float2 (&p)[4][4])
{
    for (int j = 0; j < N; ++j) {
        const float4 vj = *reinterpret_cast<const float4*>(v + j * D);
        const float4 g0 = *reinterpret_cast<const float4*>(g + j * NP);
        const float4 g1 = NQ > 2 ? *reinterpret_cast<const float4*>(g + j * NP + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float2 gq[4] = {make_float2(g0.x, g0.y), make_float2(g0.z, g0.w), make_float2(g1.x, g1.y),
                              make_float2(g1.z, g1.w)};
        const float2 vv[4] = {make_float2(vj.x, vj.x), make_float2(vj.y, vj.y), make_float2(vj.z, vj.z),
                              make_float2(vj.w, vj.w)};
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) p[q][c4] = __ffma2_rn(gq[q], vv[c4], p[q][c4]);
    }
}

// In mean mode dP[b][t] is stored already divided by the bag length L (the
// scale every lookup of the bag applies), so the per-row sums are plain sums.
template <int D, int G, typename TI>
__global__ void __launch_bounds__(G == 1 ? 128 : G * kWarp, G == 4 ? 9 : 1) interact_bwd_kernel(const __grid_constant__ BwdArgs a, float* __restrict__ dP,
                                                           int groups_per_cta)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int GT = G * kWarp;
    constexpr int CPR = D / 4;                       // float4 chunks per row
    constexpr int LPR = CPR < kWarp ? CPR : kWarp;   // lanes per row
    constexpr int CPL = CPR / LPR;                   // chunks per lane
    constexpr int RPI = kWarp / LPR;                 // row blocks worked on side by side
    const BwdLayout l = make_bwd_layout(a.T, D);
    const int group = threadIdx.x / GT;
    const int gl = threadIdx.x % GT;
    const int lane = gl % kWarp;
    const int wig = gl / kWarp;
    const int64_t b = static_cast<int64_t>(blockIdx.x) * groups_per_cta + group;
    if (b >= a.B) return;

    unsigned char* base = smem + group * l.bytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(base);
    float* V = reinterpret_cast<float*>(base + l.off_V);
    float* gm = reinterpret_cast<float*>(base + l.off_g);
    float* gos = reinterpret_cast<float*>(base + l.off_go);  // the sample's upstream row: d(out)[0..W)
    const int T = a.T, N = l.N, NP = l.NP, W = l.W;

    if (gl == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (G == 1) __syncwarp(); else __syncthreads();
    if (gl == 0) {
        const uint32_t xb = D * 4, pb = static_cast<uint32_t>(T) * D * 4;
        mbar_arrive_expect_tx(bar, xb + pb);
        bulk_g2s(V, a.dense + b * D, xb, bar);
        bulk_g2s(V + D, a.pooled + b * T * D, pb, bar);
    }
    const float* go = a.grad_out + b * W;
    for (int k = gl; k < W; k += GT) gos[k] = go[k];
    if (G == 1) __syncwarp(); else __syncthreads();
    {
        // entries e = gl, gl + GT, ... of the NP x NP matrix, (i, j) stepped without a division per entry
        const float* tri = gos + D;
        const int di = GT / NP, dj = GT - di * NP;
        int i = gl / NP, j = gl - (gl / NP) * NP;
        for (int e = gl; e < NP * NP; e += GT) {
            float v = 0.0f;
            if (i < N && j < N && i != j) v = tri[i < j ? tri_index(i, j, N) : tri_index(j, i, N)];
            gm[e] = v;
            i += di;
            j += dj;
            if (j >= NP) {
                j -= NP;
                ++i;
            }
        }
    }
    const bool landed = mbar_wait_bounded(bar, 0);
    const bool failed = (G == 1) ? (__any_sync(0xffffffffu, !landed) != 0) : (__syncthreads_or(!landed) != 0);
    if (failed) {
        if (gl == 0) {
            flag_status(a.status, DLRM_ERR_TIMEOUT);
            (void)mbar_wait_bounded(bar, 0);  // the copy still in flight ends before the group leaves
        }
        return;
    }
    if (G == 1) __syncwarp();

    const int h = lane / LPR;  // row-block lane set
    const int c0 = lane % LPR;
    const int nblk = NP / 8;
    for (int ib = wig * RPI + h; ib < nblk; ib += G * RPI) {
        const int i0 = ib * 8;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int col = (c0 + c * LPR) * 4;
            float2 p[4][4];  // p[q][c]: rows i0 + 2q, i0 + 2q + 1 at column col + c
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) p[q][c4] = make_float2(0.f, 0.f);
            // only the row pairs that hold a row of V: the last block of N = 27 has 2 of its 4
            const int nq = min(4, (N - i0 + 1) / 2);
            if (nq == 4)
                grad_rows<4>(V + col, gm + i0, N, NP, D, p);
            else if (nq == 3)
                grad_rows<3>(V + col, gm + i0, N, NP, D, p);
            else if (nq == 2)
                grad_rows<2>(V + col, gm + i0, N, NP, D, p);
            else
                grad_rows<1>(V + col, gm + i0, N, NP, D, p);
            float4 acc[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] = make_float4(p[q][0].x, p[q][1].x, p[q][2].x, p[q][3].x);
                acc[2 * q + 1] = make_float4(p[q][0].y, p[q][1].y, p[q][2].y, p[q][3].y);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = i0 + r;
                if (i >= N) break;
                if (i == 0) {
                    float4 u;
                    u.x = gos[col] + acc[0].x;
                    u.y = gos[col + 1] + acc[0].y;
                    u.z = gos[col + 2] + acc[0].z;
                    u.w = gos[col + 3] + acc[0].w;
                    *reinterpret_cast<float4*>(a.grad_dense + b * D + col) = u;
                } else {
                    float4 u = acc[r];
                    if (a.mean) {
                        const int64_t bag = static_cast<int64_t>(i - 1) * a.B + b;
                        const int64_t L = ld_index<TI>(a.offsets, bag + 1) - ld_index<TI>(a.offsets, bag);
                        if (L > 0) {
                            const float fl = static_cast<float>(L);
                            u = make_float4(__fdiv_rn(u.x, fl), __fdiv_rn(u.y, fl), __fdiv_rn(u.z, fl),
                                            __fdiv_rn(u.w, fl));
                        }
                    }
                    *reinterpret_cast<float4*>(dP + (b * T + (i - 1)) * D + col) = u;
                }
            }
        }
    }
}

// A given pooled gradient in mean mode: dP[b][t] = grad_pooled[b][t] / L(t,b),
// each element one correctly rounded division, as the interaction backward
// does it; the per-row sums then stay plain sums.  One thread per 16 bytes.
template <typename TI>
__global__ void __launch_bounds__(256) scale_by_bag_length_kernel(const __grid_constant__ BwdArgs a,
                                                                  const float* __restrict__ src,
                                                                  float* __restrict__ dst, int D)
{
    const int64_t n4 = a.B * a.T * (D / 4);
    for (int64_t e = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; e < n4; e += int64_t{gridDim.x} * blockDim.x) {
        const int64_t row = e / (D / 4);  // b * T + t
        const int64_t b = row / a.T, t = row - b * a.T;
        const int64_t bag = t * a.B + b;
        const int64_t L = ld_index<TI>(a.offsets, bag + 1) - ld_index<TI>(a.offsets, bag);
        float4 v = reinterpret_cast<const float4*>(src)[e];
        if (L > 0) {
            const float fl = static_cast<float>(L);
            v = make_float4(__fdiv_rn(v.x, fl), __fdiv_rn(v.y, fl), __fdiv_rn(v.z, fl), __fdiv_rn(v.w, fl));
        }
        reinterpret_cast<float4*>(dst)[e] = v;
    }
}

// ---------------------------------------------------------------------------
// 2. Lookup keys: key = global row id (row_base[t] + index), value = the dP
// row of the lookup's bag (b*T + t).  Lookups that update nothing keep the
// sentinel key (written first by a fill), which sorts last.
// ---------------------------------------------------------------------------
__global__ void fill_u32_kernel(uint32_t* p, int64_t n, uint32_t v)
{
    for (int64_t i = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; i < n; i += int64_t{gridDim.x} * blockDim.x)
        p[i] = v;
}

// Each warp takes 32 consecutive bags (table-major order, so the lookups of
// those bags are one contiguous range of positions) and walks the range with
// consecutive lanes on consecutive positions.  A lane finds the bag of its
// position p among the warp's 32 as the number of bags that end at or before
// p (bag ends are non-decreasing), by a 5-step search over the lanes' ends.
template <typename TI>
__global__ void __launch_bounds__(256) expand_keys_kernel(const __grid_constant__ BwdArgs a,
                                                          uint32_t* __restrict__ keys, uint32_t* __restrict__ vals)
{
    const int64_t nbags = static_cast<int64_t>(a.T) * a.B;
    const int lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (ld_index<TI>(a.offsets, 0) != 0 || ld_index<TI>(a.offsets, nbags) != a.nnz)
            flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
    }
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / kWarp);
    for (int64_t bag0 = (static_cast<int64_t>(blockIdx.x) * (blockDim.x / kWarp) + threadIdx.x / kWarp) * kWarp;
         bag0 < nbags; bag0 += warps * kWarp) {
        const int64_t bag = bag0 + lane;
        const bool live = bag < nbags;
        const int64_t s0 = live ? ld_index<TI>(a.offsets, bag) : 0;
        const int64_t s1 = live ? ld_index<TI>(a.offsets, bag + 1) : 0;
        if (__any_sync(0xffffffffu, live && (s0 < 0 || s1 < s0 || s1 > a.nnz))) {
            if (lane == 0) flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
            continue;  // the warp's positions keep the sentinel key
        }
        const int last = static_cast<int>(min(static_cast<int64_t>(kWarp - 1), nbags - 1 - bag0));
        const int64_t begin = __shfl_sync(0xffffffffu, s0, 0);
        const int64_t end = __shfl_sync(0xffffffffu, s1, last);
        const int64_t e = live ? s1 : INT64_MAX;  // bag ends; lanes past the last bag end never
        const int t = live ? static_cast<int>(bag / a.B) : 0;
        const uint32_t v = live ? static_cast<uint32_t>((bag - int64_t{t} * a.B) * a.T + t) : 0u;
        const int64_t rb = a.row_base[t], nr = a.num_rows[t];
        for (int64_t p = begin + lane; __any_sync(0xffffffffu, p < end); p += kWarp) {
            int at = 0;  // bags of this warp that end at or before p
#pragma unroll
            for (int step = 16; step >= 1; step >>= 1)
                if (__shfl_sync(0xffffffffu, e, at + step - 1) <= p) at += step;
            const uint32_t pv = __shfl_sync(0xffffffffu, v, at);
            const int64_t prb = __shfl_sync(0xffffffffu, rb, at), pnr = __shfl_sync(0xffffffffu, nr, at);
            if (p < end) {
                const int64_t r = ld_index<TI>(a.indices, p);
                if (r < 0 || r >= pnr) {
                    flag_status(a.status, DLRM_ERR_INDEX_OOB);
                } else {
                    keys[p] = static_cast<uint32_t>(prb + r);
                    vals[p] = pv;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 3. Stable LSD radix sort of (key, value) pairs by key, up to 9 bits per pass
//    (digits of `dbits` bits, bins = 2^dbits):
//    hist:    digit counts per tile of 4096 pairs   -> counts[digit][tile]
//    scan:    per digit, exclusive scan over tiles; digit totals
//    scatter: rank each pair among equal digits of its tile (earlier
//             positions first), reorder the tile by digit in shared memory,
//             then write each digit's run to its place: digit base + tile
//             offset, so neighbouring threads write neighbouring positions.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSortThreads) radix_hist_kernel(const uint32_t* __restrict__ keys, int64_t n,
                                                                  int shift, int dbits, uint32_t* __restrict__ counts,
                                                                  int64_t num_tiles)
{
    __shared__ uint32_t h[kMaxBins];
    const int bins = 1 << dbits;
    const uint32_t dmask = static_cast<uint32_t>(bins - 1);
    for (int i = threadIdx.x; i < bins; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const int64_t tile = blockIdx.x;
    const int64_t t0 = tile * kSortTile;
    uint32_t k[kSortItems];
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {  // every load in flight first
        const int64_t p = t0 + i * kSortThreads + threadIdx.x;
        k[i] = p < n ? keys[p] : 0u;
    }
#pragma unroll
    for (int i = 0; i < kSortItems; ++i)
        if (t0 + i * kSortThreads + threadIdx.x < n) atomicAdd(&h[(k[i] >> shift) & dmask], 1u);
    __syncthreads();
    for (int d = threadIdx.x; d < bins; d += blockDim.x) counts[d * num_tiles + tile] = h[d];
}

// One CTA per digit: in-place exclusive scan of counts[digit][0..num_tiles),
// each thread taking 8 consecutive tiles per step (2048 tiles a step).
__global__ void __launch_bounds__(256) radix_scan_kernel(uint32_t* __restrict__ counts, int64_t num_tiles,
                                                         uint32_t* __restrict__ bin_total)
{
    constexpr int IT = 8;
    __shared__ uint32_t warp_sum[8];
    uint32_t* row = counts + blockIdx.x * num_tiles;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t carry = 0;  // the same in every thread
    for (int64_t base = 0; base < num_tiles; base += 256 * IT) {
        const int64_t i0 = base + static_cast<int64_t>(threadIdx.x) * IT;
        uint32_t v[IT];
        uint32_t own = 0;
#pragma unroll
        for (int j = 0; j < IT; ++j) {
            v[j] = i0 + j < num_tiles ? row[i0 + j] : 0u;
            own += v[j];
        }
        uint32_t x = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[warp] = x;
        __syncthreads();
        uint32_t before = carry, step = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t ws = warp_sum[w];
            if (w < warp) before += ws;
            step += ws;
        }
        uint32_t run = before + x - own;  // exclusive prefix of this thread's first tile
#pragma unroll
        for (int j = 0; j < IT; ++j) {
            if (i0 + j < num_tiles) row[i0 + j] = run;
            run += v[j];
        }
        carry += step;
        __syncthreads();  // warp_sum is rewritten by the next step
    }
    if (threadIdx.x == 0) bin_total[blockIdx.x] = carry;
}

// Exclusive scan, in place, of v[0..kMaxBins) by the 256 threads of a block
// (two consecutive entries per thread); returns nothing, v holds the prefixes.
__device__ __forceinline__ void block_exclusive_scan_bins(uint32_t* v, uint32_t* wsum)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t a0 = v[2 * threadIdx.x], a1 = v[2 * threadIdx.x + 1];
    const uint32_t pair = a0 + a1;
    uint32_t x = pair;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, s);
        if (lane >= s) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    const uint32_t excl = before + x - pair;
    __syncthreads();
    v[2 * threadIdx.x] = excl;
    v[2 * threadIdx.x + 1] = excl + a0;
    __syncthreads();
}

struct ScatterSmem {
    uint32_t warp_cnt[kSortThreads / kWarp][kMaxBins];  // per warp digit counts, then their prefixes
    uint32_t base_of[kMaxBins];                          // global position of the tile's first pair of a digit
    uint32_t tile_start[kMaxBins];                       // position of a digit's first pair in the reordered tile
    uint32_t wsum[kSortThreads / kWarp];
    uint32_t key[kSortTile];
    uint32_t val[kSortTile];
};

__global__ void __launch_bounds__(kSortThreads, 2) radix_scatter_kernel(
    const uint32_t* __restrict__ keys_in, const uint32_t* __restrict__ vals_in, uint32_t* __restrict__ keys_out,
    uint32_t* __restrict__ vals_out, int64_t n, int shift, int dbits, const uint32_t* __restrict__ counts,
    int64_t num_tiles, const uint32_t* __restrict__ bin_total)
{
    constexpr int kWarps = kSortThreads / kWarp;
    constexpr int kPerWarp = kSortTile / kWarps;  // consecutive pairs per warp
    extern __shared__ __align__(16) unsigned char sort_smem[];
    ScatterSmem& sm = *reinterpret_cast<ScatterSmem*>(sort_smem);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t tile = blockIdx.x;
    const int bins = 1 << dbits;
    const uint32_t dmask = static_cast<uint32_t>(bins - 1);
    const int64_t t0 = tile * kSortTile;
    const int tile_n = static_cast<int>(min(static_cast<int64_t>(kSortTile), n - t0));

    // every global load of the thread first: its pairs, two digit totals, two tile offsets
    const int64_t w0 = t0 + warp * kPerWarp;
    uint32_t key[kPerWarp / kWarp], val[kPerWarp / kWarp], rank[kPerWarp / kWarp];
#pragma unroll
    for (int r = 0; r < kPerWarp / kWarp; ++r) {
        const int64_t p = w0 + r * kWarp + lane;
        key[r] = p < n ? keys_in[p] : 0u;
        val[r] = p < n ? vals_in[p] : 0u;
    }
    uint32_t tot[2], off[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int d = 2 * threadIdx.x + j;
        tot[j] = d < bins ? bin_total[d] : 0u;
        off[j] = d < bins ? counts[d * num_tiles + tile] : 0u;
    }
    for (int i = threadIdx.x; i < kWarps * kMaxBins; i += blockDim.x) (&sm.warp_cnt[0][0])[i] = 0;
    // digit bases: exclusive scan of the digit totals, plus this tile's offset within each digit
#pragma unroll
    for (int j = 0; j < 2; ++j) sm.base_of[2 * threadIdx.x + j] = tot[j];
    __syncthreads();
    block_exclusive_scan_bins(sm.base_of, sm.wsum);
#pragma unroll
    for (int j = 0; j < 2; ++j) sm.base_of[2 * threadIdx.x + j] += off[j];

    // stable ranks: warp w ranks pairs w*kPerWarp .. of the tile in order, 32 at a time
    const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < kPerWarp / kWarp; ++r) {
        const int64_t p = w0 + r * kWarp + lane;
        const bool live = p < n;
        const uint32_t d = (key[r] >> shift) & dmask;
        const uint32_t live_mask = __ballot_sync(0xffffffffu, live);
        const uint32_t peers = __match_any_sync(0xffffffffu, live ? d : 0xFFFFFFFFu) & live_mask;
        const uint32_t before = sm.warp_cnt[warp][d];
        rank[r] = before + __popc(peers & lt_mask);
        __syncwarp();
        if (live && (peers & ~((lt_mask << 1) | 1u)) == 0) sm.warp_cnt[warp][d] = before + __popc(peers);  // last peer
        __syncwarp();
    }
    __syncthreads();
    // per digit: exclusive prefix over warps (warp order = position order) and the tile's digit count
    for (int d = threadIdx.x; d < kMaxBins; d += blockDim.x) {
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t c = sm.warp_cnt[w][d];
            sm.warp_cnt[w][d] = run;
            run += c;
        }
        sm.tile_start[d] = run;
    }
    __syncthreads();
    block_exclusive_scan_bins(sm.tile_start, sm.wsum);
    // the tile reordered by digit (stable), in shared memory
#pragma unroll
    for (int r = 0; r < kPerWarp / kWarp; ++r) {
        const int64_t p = w0 + r * kWarp + lane;
        if (p < n) {
            const uint32_t d = (key[r] >> shift) & dmask;
            const uint32_t at = sm.tile_start[d] + sm.warp_cnt[warp][d] + rank[r];
            sm.key[at] = key[r];
            sm.val[at] = val[r];
        }
    }
    __syncthreads();
    // each digit's run to its place: consecutive threads, consecutive positions
    for (int i = threadIdx.x; i < tile_n; i += kSortThreads) {
        const uint32_t k = sm.key[i];
        const uint32_t d = (k >> shift) & dmask;
        const uint32_t dst = sm.base_of[d] + (static_cast<uint32_t>(i) - sm.tile_start[d]);
        keys_out[dst] = k;
        vals_out[dst] = sm.val[i];
    }
}

// ---------------------------------------------------------------------------
// 4. Ordered per-row gradient sums and row-wise Adagrad.
// Sorted lookups are cut into chunks of kChunk.  One warp per chunk walks its
// lookups in order and sums dP rows run by run (a run = equal keys).  A run
// that lies inside its chunk is finished at once (Adagrad on its row).  A run
// cut by a chunk border leaves a partial sum: the chunk's first run in slot
// 2c, its last run (if different) in slot 2c+1; a second kernel adds the
// pieces of each cut run in chunk order and applies Adagrad.
// ---------------------------------------------------------------------------
// lane owns elements [4*lane, 4*lane+4) (+128 for D = 256) when D >= 128;
// for D < 128 lanes 0..D/4-1 own one float4 each.
template <int D>
struct Lanes {
    static constexpr int kChunks = D >= 128 ? D / 128 : 1;
    static constexpr int kActive = D >= 128 ? kWarp : D / 4;
};

// w - step * g, each element one fused multiply-add (as fmaf), two at a time (fma.rn.f32x2).
__device__ __forceinline__ float4 step_row(float4 w, float4 g, float step)
{
    const float2 ns = make_float2(-step, -step);
    const float2 a = __ffma2_rn(ns, make_float2(g.x, g.y), make_float2(w.x, w.y));
    const float2 b = __ffma2_rn(ns, make_float2(g.z, g.w), make_float2(w.z, w.w));
    return make_float4(a.x, a.y, b.x, b.y);
}

// g += v, elementwise, two at a time (add.f32x2: each an fp32 add rounded once).
__device__ __forceinline__ void add4(float4& g, float4 v)
{
    const float2 a = __fadd2_rn(make_float2(g.x, g.y), make_float2(v.x, v.y));
    const float2 b = __fadd2_rn(make_float2(g.z, g.w), make_float2(v.z, v.w));
    g = make_float4(a.x, a.y, b.x, b.y);
}

// One update of the row `key` of table t whose summed gradient (this lane's slice) is g:
//   Adagrad (row-wise): A += mean_d g_d^2, w -= lr g / (sqrt(A) + eps);   SGD: w -= lr g.
template <int D>
__device__ __forceinline__ void adagrad_row(const BwdArgs& a, uint32_t key, int t, const float4 (&g)[Lanes<D>::kChunks],
                                            int lane)
{
    constexpr int C = Lanes<D>::kChunks;
    const bool active = lane < Lanes<D>::kActive;
    if (a.rule == DLRM_RULE_SGD) {
        if (active) {
            float* w = a.tables[t] + (static_cast<int64_t>(key) - a.row_base[t]) * D;
#pragma unroll
            for (int k = 0; k < C; ++k) {
                const int col = (lane + k * kWarp) * 4;
                *reinterpret_cast<float4*>(w + col) = step_row(*reinterpret_cast<const float4*>(w + col), g[k], a.lr);
            }
        }
        return;
    }
    float ss = 0.0f;
    if (active) {
#pragma unroll
        for (int k = 0; k < C; ++k) ss += g[k].x * g[k].x + g[k].y * g[k].y + g[k].z * g[k].z + g[k].w * g[k].w;
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
    const int64_t r = static_cast<int64_t>(key) - a.row_base[t];
    float* acc = a.accum[t] + r;
    const float A = *acc + ss / static_cast<float>(D);
    const float step = a.lr / (sqrtf(A) + a.eps);  // one division per row
    if (active) {
        float* w = a.tables[t] + r * D;
#pragma unroll
        for (int k = 0; k < C; ++k) {
            const int col = (lane + k * kWarp) * 4;
            float4 v = *reinterpret_cast<float4*>(w + col);
            v = step_row(v, g[k], step);
            *reinterpret_cast<float4*>(w + col) = v;
        }
    }
    __syncwarp();
    if (lane == 0) *acc = A;
}

// t = v / T for v < 2^32, with magic = ceil(2^64 / T) (T >= 2): the product's
// high word (Granlund & Montgomery's division by invariant integers).
__device__ __forceinline__ uint32_t div_by_T(uint32_t v, const BwdArgs& a)
{
    return a.T == 1 ? v : static_cast<uint32_t>(__umul64hi(static_cast<uint64_t>(v), a.t_magic));
}

// The update of one row whose weights (this lane's slice) and accumulator
// were read earlier: w is the row before the step, acc_old its accumulator
// (Adagrad only).
template <int D>
__device__ __forceinline__ void adagrad_apply(const BwdArgs& a, uint32_t key, int t,
                                              const float4 (&g)[Lanes<D>::kChunks],
                                              const float4 (&w)[Lanes<D>::kChunks], float acc_old, int lane)
{
    constexpr int C = Lanes<D>::kChunks;
    const bool active = lane < Lanes<D>::kActive;
    if (a.rule == DLRM_RULE_SGD) {
        if (active) {
            float* wr = a.tables[t] + (static_cast<int64_t>(key) - a.row_base[t]) * D;
#pragma unroll
            for (int k = 0; k < C; ++k)
                *reinterpret_cast<float4*>(wr + (lane + k * kWarp) * 4) = step_row(w[k], g[k], a.lr);
        }
        return;
    }
    float ss = 0.0f;
    if (active) {
#pragma unroll
        for (int k = 0; k < C; ++k) ss += g[k].x * g[k].x + g[k].y * g[k].y + g[k].z * g[k].z + g[k].w * g[k].w;
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
    const int64_t r = static_cast<int64_t>(key) - a.row_base[t];
    const float A = acc_old + ss / static_cast<float>(D);
    const float step = a.lr / (sqrtf(A) + a.eps);  // one division per row
    if (active) {
        float* wr = a.tables[t] + r * D;
#pragma unroll
        for (int k = 0; k < C; ++k) {
            const float4 v = step_row(w[k], g[k], step);
            *reinterpret_cast<float4*>(wr + (lane + k * kWarp) * 4) = v;
        }
    }
    if (lane == 0) a.accum[t][r] = A;
}

// Shared-memory copies (cp.async: global -> shared without a register stop).
// A lane reads back only the bytes it copied itself (the accumulator aside),
// so its own cp.async.wait_group is the only wait the ring needs.
__device__ __forceinline__ void seg_copy16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void seg_copy4(void* dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void seg_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void seg_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The per-row sums keep kDepth - 1 lookups in flight per warp: each lookup's
// dP row and, where a run starts, its row's weights and accumulator travel
// into a ring of kDepth shared-memory slots while the warp walks earlier
// lookups.  A slot is refilled one lookup after it was read.
template <int D>
struct alignas(16) SegRing {
    static constexpr int kDepth = 5;
    static constexpr int kMinBlocks = D >= 256 ? 4 : 8;  // CTAs of 4 warps per SM (shared memory, registers)
    static constexpr uint8_t kNoRun = 0xFF;                 // table[] of a lookup that starts no run
    float drow[kDepth][D];   // dP rows
    float wrow[kDepth][D];   // weights of the rows whose runs start at these lookups
    float acc[kDepth];       // their accumulators (Adagrad)
    uint32_t key[kChunk];    // the chunk's sorted lookups
    uint32_t val[kChunk];
    uint8_t table[kChunk];   // the table of a run's row at the run's first lookup, kNoRun elsewhere
};

template <int D>
constexpr size_t seg_smem_bytes()
{
    return sizeof(SegRing<D>) * (kSegThreads / kWarp);
}

// One warp per chunk.  The chunk is staged once, lane-parallel: keys, values
// and, at each lookup whose key differs from the one before (a run starts),
// the table of its row.  Then the warp walks the lookups in order, adds each
// dP row into the running sum of its run and updates the row when the run
// ends inside the chunk.
template <int D>
__global__ void __launch_bounds__(kSegThreads, SegRing<D>::kMinBlocks) segment_chunk_kernel(
    const __grid_constant__ BwdArgs a, const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals,
    const float* __restrict__ dP, float* __restrict__ partial, int64_t num_chunks)
{
    constexpr int C = Lanes<D>::kChunks;
    constexpr int R = SegRing<D>::kDepth;
    constexpr uint8_t kNoRun = SegRing<D>::kNoRun;
    extern __shared__ __align__(16) unsigned char seg_smem[];
    const int lane = threadIdx.x & 31;
    const int64_t chunk = blockIdx.x * int64_t{blockDim.x / kWarp} + (threadIdx.x >> 5);
    if (chunk >= num_chunks) return;
    SegRing<D>& ring = reinterpret_cast<SegRing<D>*>(seg_smem)[threadIdx.x >> 5];
    const bool active = lane < Lanes<D>::kActive;
    const int64_t c0 = chunk * kChunk;
    const int n = static_cast<int>(min(static_cast<int64_t>(kChunk), a.nnz - c0));
    const uint32_t before_key = c0 > 0 ? keys[c0 - 1] : kSentinel;
    const uint32_t after_key = c0 + n < a.nnz ? keys[c0 + n] : kSentinel;

    // lookups that update nothing (sentinel keys) sort last, so the live ones are a prefix
    int live = 0;
    uint32_t prev = before_key;
    for (int i0 = 0; i0 < n; i0 += kWarp) {
        const int i = i0 + lane;
        const uint32_t k = i < n ? keys[c0 + i] : kSentinel;
        const uint32_t v = i < n ? vals[c0 + i] : 0u;
        uint32_t kp = __shfl_up_sync(0xffffffffu, k, 1);
        if (lane == 0) kp = prev;
        prev = __shfl_sync(0xffffffffu, k, kWarp - 1);
        if (i < n) {
            ring.key[i] = k;
            ring.val[i] = v;
            ring.table[i] = k != kSentinel && k != kp
                                ? static_cast<uint8_t>(v - div_by_T(v, a) * static_cast<uint32_t>(a.T))
                                : kNoRun;
        }
        live += __popc(__ballot_sync(0xffffffffu, k != kSentinel));
    }
    __syncwarp();

    auto issue = [&](int j, int slot) {
        if (j < live) {
            if (active) {
                const float* src = dP + static_cast<int64_t>(ring.val[j]) * D;
#pragma unroll
                for (int q = 0; q < C; ++q) {
                    const int col = (lane + q * kWarp) * 4;
                    seg_copy16(&ring.drow[slot][col], src + col);
                }
            }
            const int t = ring.table[j];
            if (t != kNoRun) {  // a run starts here: its row's weights and accumulator too
                const int64_t r = static_cast<int64_t>(ring.key[j]) - a.row_base[t];
                if (active) {
                    const float* wr = a.tables[t] + r * D;
#pragma unroll
                    for (int q = 0; q < C; ++q) {
                        const int col = (lane + q * kWarp) * 4;
                        seg_copy16(&ring.wrow[slot][col], wr + col);
                    }
                }
                if (lane == 0 && a.rule == DLRM_RULE_ADAGRAD) seg_copy4(&ring.acc[slot], a.accum[t] + r);
            }
        }
        seg_commit();  // one group per lookup, empty past the end, so the wait below counts lookups
    };

    uint32_t cur = kSentinel;
    int cur_t = 0;
    bool cur_first = true;  // current run is the chunk's first run
    float4 g[C], cw[C];     // the run's gradient sum; its row's weights
    float ca = 0.0f;        // its accumulator
#pragma unroll
    for (int q = 0; q < C; ++q) g[q] = cw[q] = make_float4(0.f, 0.f, 0.f, 0.f);

    auto flush = [&]() {
        if (cur == kSentinel) return;
        const bool cut_before = cur_first && before_key == cur;
        const bool cut_after = after_key == cur;
        if (!cut_before && !cut_after) {
            adagrad_apply<D>(a, cur, cur_t, g, cw, ca, lane);
        } else {
            float* dst = partial + ((chunk * 2) + (cur_first ? 0 : 1)) * D;
            if (active) {
#pragma unroll
                for (int q = 0; q < C; ++q) *reinterpret_cast<float4*>(dst + (lane + q * kWarp) * 4) = g[q];
            }
        }
    };

#pragma unroll
    for (int j = 0; j < R - 1; ++j) issue(j, j);
    int rs = 0, ws = R - 1;  // the slot read now, the slot refilled now
#pragma unroll 2
    for (int j = 0; j < live; ++j) {
        seg_wait<R - 2>();  // this lookup's group has landed
        const int t = ring.table[j];
        if (t != kNoRun || j == 0) {  // a run starts (j == 0 may continue a run cut at the chunk's start)
            flush();
            cur_first = j == 0;
            cur = ring.key[j];
            cur_t = t;
            if (t != kNoRun) {
                if (a.rule == DLRM_RULE_ADAGRAD) {
                    __syncwarp();  // lane 0's accumulator copy, landed, is seen by the warp
                    ca = ring.acc[rs];
                    __syncwarp();  // and read by every lane before lane 0 refills the slot
                }
#pragma unroll
                for (int q = 0; q < C; ++q)
                    if (active) cw[q] = *reinterpret_cast<const float4*>(&ring.wrow[rs][(lane + q * kWarp) * 4]);
            }
#pragma unroll
            for (int q = 0; q < C; ++q) g[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (active) {
#pragma unroll
            for (int q = 0; q < C; ++q) add4(g[q], *reinterpret_cast<const float4*>(&ring.drow[rs][(lane + q * kWarp) * 4]));
        }
        issue(j + R - 1, ws);  // refills the slot read one lookup ago
        rs = rs + 1 == R ? 0 : rs + 1;
        ws = ws + 1 == R ? 0 : ws + 1;
    }
    seg_wait<0>();
    flush();
}

// One warp per chunk that holds the start of a run cut by its end border.
template <int D>
__global__ void __launch_bounds__(kSegThreads) segment_span_kernel(const __grid_constant__ BwdArgs a,
                                                           const uint32_t* __restrict__ keys,
                                                           const uint32_t* __restrict__ vals,
                                                           const float* __restrict__ partial, int64_t num_chunks)
{
    constexpr int C = Lanes<D>::kChunks;
    const int lane = threadIdx.x & 31;
    const int64_t chunk = blockIdx.x * int64_t{blockDim.x / kWarp} + (threadIdx.x >> 5);
    if (chunk >= num_chunks) return;
    const bool active = lane < Lanes<D>::kActive;
    const int64_t c0 = chunk * kChunk;
    const int64_t c1 = min(c0 + kChunk, a.nnz);
    if (c1 >= a.nnz) return;  // last chunk: nothing runs past it
    const uint32_t key = keys[c1 - 1];
    if (key == kSentinel || keys[c1] != key) return;     // last run not cut
    const bool whole = keys[c0] == key;                   // chunk is one run
    if (whole && c0 > 0 && keys[c0 - 1] == key) return;   // run started in an earlier chunk
    const uint32_t v_last = vals[c1 - 1];
    const int t = static_cast<int>(v_last - div_by_T(v_last, a) * static_cast<uint32_t>(a.T));

    // the run holds a piece of every later chunk whose first key is its key: those chunks are
    // consecutive; find the last, 32 chunk borders at a time
    int64_t last = chunk;
    for (int64_t cb = chunk + 1;; cb += kWarp) {
        const int64_t c = cb + lane;
        const bool piece = c < num_chunks && keys[c * kChunk] == key;
        const uint32_t m = __ballot_sync(0xffffffffu, piece);
        const int n = m == 0xffffffffu ? kWarp : __ffs(~m) - 1;  // leading pieces
        last = cb + n - 1;
        if (n < kWarp) break;
    }

    // partial sums added in chunk order (the reproducible order), 8 in flight
    float4 g[C];
#pragma unroll
    for (int k = 0; k < C; ++k) g[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](const float4 (&v)[C]) {
#pragma unroll
        for (int k = 0; k < C; ++k) add4(g[k], v[k]);
    };
    auto load = [&](int64_t slot, float4 (&v)[C]) {
        const float* src = partial + slot * D;
#pragma unroll
        for (int k = 0; k < C; ++k) v[k] = *reinterpret_cast<const float4*>(src + (lane + k * kWarp) * 4);
    };
    if (active) {
        float4 first[C];
        load(chunk * 2 + (whole ? 0 : 1), first);
        add(first);
        for (int64_t c = chunk + 1; c <= last; c += 8) {
            float4 v[8][C];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + u <= last) load((c + u) * 2, v[u]);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + u <= last) add(v[u]);
        }
    }
    adagrad_row<D>(a, key, t, g, lane);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
constexpr int kMaxSmem = 227 * 1024;

template <int D, int G, typename TI>
dlrm_status launch_interact_bwd(const BwdArgs& a, float* dP, cudaStream_t s)
{
    const BwdLayout l = make_bwd_layout(a.T, D);
    int groups = 1;
    if (G == 1) {
        groups = kMaxSmem / l.bytes;
        if (groups > 4) groups = 4;
        if (groups < 1) return DLRM_ERR_UNSUPPORTED;
    } else if (l.bytes > kMaxSmem) {
        return DLRM_ERR_UNSUPPORTED;
    }
    const size_t smem = static_cast<size_t>(groups) * l.bytes;
    auto kern = interact_bwd_kernel<D, G, TI>;
    if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) != cudaSuccess)
        return DLRM_ERR_CUDA;
    const int64_t blocks = (a.B + groups - 1) / groups;
    kern<<<static_cast<unsigned>(blocks), groups * G * kWarp, smem, s>>>(a, dP, groups);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

// Key bits: valid keys are < total rows, so the sentinel's low bits sort after them; the passes split
// them into digits of at most kMaxRadixBits bits.  The sorted pairs end in ping-pong buffer passes % 2.
void radix_digits(const BwdArgs& a, int* passes, int* dbits)
{
    int bits = 1;
    while ((int64_t{1} << bits) <= a.row_base[a.T]) ++bits;
    *passes = (bits + kMaxRadixBits - 1) / kMaxRadixBits;
    *dbits = (bits + *passes - 1) / *passes;
}

// Keys, then the stable radix sort, on stream ks; returns the ping-pong buffer holding the sorted pairs.
template <typename TI>
dlrm_status sort_keys(const BwdArgs& a, const Workspace& w, cudaStream_t ks, int* sorted)
{
    const int64_t nbags = int64_t{a.T} * a.B;
    fill_u32_kernel<<<148 * 8, 256, 0, ks>>>(w.keys[0], a.nnz, kSentinel);
    const int64_t expand_blocks = (nbags + 255) / 256;  // a warp per 32 bags
    expand_keys_kernel<TI><<<static_cast<unsigned>(expand_blocks < 148 * 64 ? expand_blocks : 148 * 64), 256, 0, ks>>>(
        a, w.keys[0], w.vals[0]);

    int passes = 0, dbits = 0;
    radix_digits(a, &passes, &dbits);
    // set on every call: the attribute belongs to the current device's context
    if (cudaFuncSetAttribute(radix_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(ScatterSmem))) != cudaSuccess)
        return DLRM_ERR_CUDA;
    int cur = 0;
    for (int pass = 0; pass < passes; ++pass) {
        const int shift = pass * dbits;
        radix_hist_kernel<<<static_cast<unsigned>(w.num_tiles), kSortThreads, 0, ks>>>(w.keys[cur], a.nnz, shift,
                                                                                      dbits, w.counts, w.num_tiles);
        radix_scan_kernel<<<1u << dbits, 256, 0, ks>>>(w.counts, w.num_tiles, w.bin_total);
        radix_scatter_kernel<<<static_cast<unsigned>(w.num_tiles), kSortThreads, sizeof(ScatterSmem), ks>>>(
            w.keys[cur], w.vals[cur], w.keys[cur ^ 1], w.vals[cur ^ 1], a.nnz, shift, dbits, w.counts, w.num_tiles,
            w.bin_total);
        cur ^= 1;
    }
    *sorted = cur;
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

// The lookup keys can be built and sorted on a second stream while the
// interaction backward runs on the caller's stream: the two read the same
// inputs and write disjoint parts of the workspace, and only the per-row sums
// need both.  The caller supplies that stream (the library owns none); fork
// and join are two events made for this call and released once queued, so
// calls on independent streams share nothing, and the pattern also holds
// while the caller's stream is being captured into a CUDA graph.
struct Fork {
    cudaEvent_t fork = nullptr, join = nullptr;
    ~Fork()
    {
        // an event destroyed after being queued is released once the device has passed it
        if (fork) cudaEventDestroy(fork);
        if (join) cudaEventDestroy(join);
    }
};

template <int D, typename TI>
dlrm_status launch_interact_bwd_groups(const BwdArgs& a, float* dP, cudaStream_t s)
{
    // warps per sample: one per 8-row block of dV up to 4 (N <= 32), else 8; a sample's V is staged once
    const int nblk = round_up(a.T + 1, 8) / 8;
    return nblk > 4   ? launch_interact_bwd<D, 8, TI>(a, dP, s)
           : nblk > 2 ? launch_interact_bwd<D, 4, TI>(a, dP, s)
                      : launch_interact_bwd<D, 1, TI>(a, dP, s);
}

// The training step (source kFromInteraction: dP from the interaction backward, already divided by the
// bag lengths in mean mode) or the row update from a given pooled gradient (kFromPooledGrad).
// presorted: the workspace holds the sorted pairs of these bags (sort_keys queued earlier by the caller),
// so only the dP rows and the per-row sums run here; the per-row sums wait for `sorted` when it is given.
// grad_ready, if given, is recorded on s once the interaction backward (grad_dense, dP) is queued.
template <int D, typename TI>
dlrm_status run_backward(const BwdArgs& a, const Workspace& w, int source, const float* grad_pooled, cudaStream_t s,
                         cudaStream_t side, bool presorted, cudaEvent_t sorted, cudaEvent_t grad_ready)
{
    Fork f;
    const bool two = !presorted && side != nullptr && side != s && a.nnz > 0;
    if (two && (cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventRecord(f.fork, s) != cudaSuccess || cudaStreamWaitEvent(side, f.fork, 0) != cudaSuccess))
        return DLRM_ERR_CUDA;
    const cudaStream_t ks = two ? side : s;

    int cur = 0;
    dlrm_status st = DLRM_OK;
    if (presorted) {
        int passes = 0, dbits = 0;
        radix_digits(a, &passes, &dbits);
        cur = passes & 1;
    } else if (a.nnz > 0) {
        st = sort_keys<TI>(a, w, ks, &cur);
    }
    // beside the sort: the dP rows the per-row sums read
    const float* dP = source == kFromInteraction ? w.dP : grad_pooled;
    if (st == DLRM_OK) {
        if (source == kFromInteraction) {
            st = launch_interact_bwd_groups<D, TI>(a, w.dP, s);
            if (st == DLRM_OK && grad_ready != nullptr && cudaEventRecord(grad_ready, s) != cudaSuccess)
                st = DLRM_ERR_CUDA;
        } else if (a.mean && a.nnz > 0) {
            const int64_t n4 = a.B * a.T * (D / 4);
            const int64_t blocks = (n4 + 255) / 256;
            scale_by_bag_length_kernel<TI><<<static_cast<unsigned>(blocks < 148 * 16 ? blocks : 148 * 16), 256, 0, s>>>(
                a, grad_pooled, w.dP, D);
            dP = w.dP;
            st = cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
        }
    }
    // the side stream's work joins the caller's stream whatever happened above
    if (two && (cudaEventRecord(f.join, side) != cudaSuccess || cudaStreamWaitEvent(s, f.join, 0) != cudaSuccess))
        return DLRM_ERR_CUDA;
    if (st != DLRM_OK || a.nnz == 0) return st;
    if (presorted && sorted != nullptr && cudaStreamWaitEvent(s, sorted, 0) != cudaSuccess) return DLRM_ERR_CUDA;

    const unsigned seg_blocks = static_cast<unsigned>((w.num_chunks + kSegThreads / kWarp - 1) / (kSegThreads / kWarp));
    constexpr size_t seg_smem = seg_smem_bytes<D>();
    if (seg_smem > 48 * 1024 &&
        cudaFuncSetAttribute(segment_chunk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(seg_smem)) != cudaSuccess)
        return DLRM_ERR_CUDA;
    segment_chunk_kernel<D><<<seg_blocks, kSegThreads, seg_smem, s>>>(a, w.keys[cur], w.vals[cur], dP, w.partial,
                                                                      w.num_chunks);
    segment_span_kernel<D><<<seg_blocks, kSegThreads, 0, s>>>(a, w.keys[cur], w.vals[cur], w.partial, w.num_chunks);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

template <int D>
dlrm_status dispatch_bwd(const BwdArgs& a, int index_type, const Workspace& w, int source, const float* grad_pooled,
                         cudaStream_t s, cudaStream_t side, bool presorted, cudaEvent_t sorted, cudaEvent_t grad_ready)
{
    return index_type == DLRM_I32
               ? run_backward<D, int32_t>(a, w, source, grad_pooled, s, side, presorted, sorted, grad_ready)
               : run_backward<D, int64_t>(a, w, source, grad_pooled, s, side, presorted, sorted, grad_ready);
}

bool with_dP(int source, bool mean) { return source == kFromInteraction || mean; }

}  // namespace

size_t bwd_workspace_bytes(int64_t B, int32_t T, int32_t D, int64_t nnz, int source, bool mean)
{
    size_t total = 0;
    carve(nullptr, B, T, D, nnz, with_dP(source, mean), &total);
    return total;
}

dlrm_status launch_backward(const BwdArgs& a, int dim, int index_type, int source, const float* grad_pooled,
                            void* workspace, size_t workspace_bytes, cudaStream_t s, cudaStream_t side, bool presorted,
                            cudaEvent_t sorted, cudaEvent_t grad_ready)
{
    size_t need = 0;
    const Workspace w = carve(workspace, a.B, a.T, dim, a.nnz, with_dP(source, a.mean != 0), &need);
    if (workspace_bytes < need) return DLRM_ERR_INVALID_ARG;
    switch (dim) {
        case 16: return dispatch_bwd<16>(a, index_type, w, source, grad_pooled, s, side, presorted, sorted, grad_ready);
        case 32: return dispatch_bwd<32>(a, index_type, w, source, grad_pooled, s, side, presorted, sorted, grad_ready);
        case 64: return dispatch_bwd<64>(a, index_type, w, source, grad_pooled, s, side, presorted, sorted, grad_ready);
        case 128: return dispatch_bwd<128>(a, index_type, w, source, grad_pooled, s, side, presorted, sorted, grad_ready);
        case 256: return dispatch_bwd<256>(a, index_type, w, source, grad_pooled, s, side, presorted, sorted, grad_ready);
        default: return DLRM_ERR_UNSUPPORTED;
    }
}

dlrm_status launch_sort(const BwdArgs& a, int dim, int index_type, void* workspace, size_t workspace_bytes,
                        cudaStream_t s)
{
    if (dim != 16 && dim != 32 && dim != 64 && dim != 128 && dim != 256) return DLRM_ERR_UNSUPPORTED;
    size_t need = 0;
    const Workspace w = carve(workspace, a.B, a.T, dim, a.nnz, with_dP(kFromInteraction, a.mean != 0), &need);
    if (workspace_bytes < need) return DLRM_ERR_INVALID_ARG;
    if (a.nnz == 0) return DLRM_OK;
    int cur = 0;
    return index_type == DLRM_I32 ? sort_keys<int32_t>(a, w, s, &cur) : sort_keys<int64_t>(a, w, s, &cur);
}

dlrm_status launch_interact_backward(const BwdArgs& a, int dim, float* grad_pooled, cudaStream_t s)
{
    // no bag lengths are applied (a.mean is 0), so the offsets are never read
    switch (dim) {
        case 16: return launch_interact_bwd_groups<16, int32_t>(a, grad_pooled, s);
        case 32: return launch_interact_bwd_groups<32, int32_t>(a, grad_pooled, s);
        case 64: return launch_interact_bwd_groups<64, int32_t>(a, grad_pooled, s);
        case 128: return launch_interact_bwd_groups<128, int32_t>(a, grad_pooled, s);
        case 256: return launch_interact_bwd_groups<256, int32_t>(a, grad_pooled, s);
        default: return DLRM_ERR_UNSUPPORTED;
    }
}

}  // namespace dlrm
