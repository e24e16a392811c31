// fwd_tc.cu -- the fused sparse forward with the interaction on the tensor
// cores (tcgen05, fp32 accumulators in TMEM).
//
//   lookup + pooling        "DLRM" (robocikowo.com), "Forward pass" step (2);
//                           bags of several IDs: "The embedding table is the model"
//   N x N dot products,     same page, step (3): all vectors as rows of one
//   strict upper triangle   matrix, pairwise dot products, the N(N-1)/2 values
//                           above the diagonal
//   concatenation           same page, step (4), dense vector first
//
// Tiling.  A CTA works on tiles of 128 rows of V, the M and N of one MMA.
// A sample owns NP consecutive rows (NP = N rounded up to 32, 64 or 128):
// row 0 is the dense vector x, rows 1..T the pooled bags, the rest unused, so
// a tile holds S = 128 / NP samples.  Warp w gathers tile rows 32w..32w+31
// and later reads the same rows of the Gram back from its quarter of TMEM.
//
// Gather.  Rows with a single source (x, bags of one lookup, the pooled
// inputs of the interaction-only call) are copied by 16-byte cp.async
// straight into the operand lines, every such row of the warp in flight at
// once.  In the multi-lookup variant (bags of more than 1.25 lookups on
// average) a warp flattens the lookups of its other rows into one list and
// loads them 16 at a time (each lane a 16-byte slice of a row, the warp one
// whole row per load instruction), each added into its row in lookup order in
// fp32 (packed adds, each rounded as a scalar add).  A finished row (the
// pooled vector) is written once, as a pair of bf16 (hi = bf16(v),
// lo = bf16(v - hi)) into two K-major, 128-byte-swizzled operand buffers in
// shared memory, and to pooled_save when asked.  x is also staged exactly for
// the output row.
//
// Gram.  One thread issues, for the tile, hi*hi^T + hi*lo^T + lo*hi^T as
// 3 x D/16 MMAs of 128 x 128 x 16 into one 128 x 128 fp32 accumulator in
// TMEM (the three products keep ~16 significant bits of each operand: the
// dropped lo*lo term and the bf16 rounding of lo are below 2^-16 relative to
// sum |V_i[d] V_j[d]|).  The products of rows of different samples are
// computed and never read; at N <= 32 that is 3/4 of the tile.
//
// Epilogue.  Each warp loads its rows of its sample's diagonal block from TMEM
// (thread i gets row i of the Gram), scatters the values above the diagonal
// into the staged output row, and the CTA stores the tile's output rows with
// coalesced stores.  A one-sample tile (N > 64: a triangle of up to 8,001
// values) instead leaves through one bulk copy of the TMA engine, issued by
// one thread, while the warps go on to the next tile; its x went straight to
// out when it was split.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dlrm {
namespace {

constexpr int kTileRows = 128;      // rows of V per tile: the MMA's M and N
constexpr int kThreads = 128;       // 4 warps; warp w owns tile rows [32w, 32w + 32)
constexpr int kTmemCols = 128;      // one 128 x 128 fp32 accumulator
constexpr int kMaxCtasPerSm = 4;    // 4 x 128 TMEM columns fill the SM's 512
constexpr int kMinSmemPerCta = 48 * 1024;  // keeps at most 4 CTAs on an SM
constexpr uint32_t kFull = 0xffffffffu;

// Floats between the staged triangles of a tile's samples: room for W - D values placed at the 16-byte
// residue of their place in out (up to 3 floats in), each slot 16-byte aligned.
__host__ __device__ constexpr int stage_stride(int D, int W) { return (W - D + 3 + 3) & ~3; }

// Shared memory of one CTA, byte offsets from a 1024-byte aligned base.
struct TcLayout {
    int hi, lo, stage, tables, bar, tmem_slot, bytes;
};

constexpr int kMaxTablesTc = kTileRows - 1;  // N = T + 1 <= 128

__host__ __device__ inline TcLayout make_tc_layout(int D, int S, int W)
{
    TcLayout l;
    const int operand = kTileRows * D * 2;  // one bf16 operand
    l.hi = 0;
    l.lo = operand;
    l.stage = 2 * operand;  // S output rows of W floats; one-sample tiles: the triangle alone (stage_stride)
    l.tables = l.stage + (S == 1 ? stage_stride(D, W) * 4 : round_up(S * W * 4, 16));  // table addresses, rows
    l.bar = l.tables + 16 * kMaxTablesTc;
    l.tmem_slot = l.bar + 8;  // after the MMA barrier
    l.bytes = l.tmem_slot + 16;
    return l;
}

template <typename TI>
__device__ __forceinline__ int64_t load_idx(const void* p, int64_t i)
{
    return static_cast<int64_t>(__ldg(static_cast<const TI*>(p) + i));
}

__device__ __forceinline__ int64_t shfl64(int64_t v, int src)
{
    const int lo = __shfl_sync(kFull, static_cast<int>(v & 0xffffffff), src);
    const int hi = __shfl_sync(kFull, static_cast<int>(v >> 32), src);
    return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

// One lane's slice of a row: C elements of type TE.
template <int BYTES>
struct Slice;
template <>
struct Slice<16> {
    uint4 v;
    __device__ __forceinline__ void load(const void* row, int lane) { v = __ldg(static_cast<const uint4*>(row) + lane); }
    __device__ __forceinline__ uint32_t w(int i) const { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
};
template <>
struct Slice<8> {
    uint2 v;
    __device__ __forceinline__ void load(const void* row, int lane) { v = __ldg(static_cast<const uint2*>(row) + lane); }
    __device__ __forceinline__ uint32_t w(int i) const { return i == 0 ? v.x : v.y; }
};
template <>
struct Slice<4> {
    uint32_t v;
    __device__ __forceinline__ void load(const void* row, int lane) { v = __ldg(static_cast<const uint32_t*>(row) + lane); }
    __device__ __forceinline__ uint32_t w(int) const { return v; }
};

// Widen a slice to fp32 (bf16 is the upper half of an fp32 pattern: exact).
template <int C, typename TE, typename SL>
__device__ __forceinline__ void widen(const SL& s, float (&f)[C])
{
    if constexpr (sizeof(TE) == 4) {
#pragma unroll
        for (int c = 0; c < C; ++c) f[c] = __uint_as_float(s.w(c));
    } else {
#pragma unroll
        for (int i = 0; i < C / 2; ++i) {
            const uint32_t x = s.w(i);
            f[2 * i] = __uint_as_float(x << 16);
            f[2 * i + 1] = __uint_as_float(x & 0xffff0000u);
        }
    }
}

// Byte offset of (row, byte b of the row's K extent) in a K-major operand of
// kTileRows rows in the 128-byte swizzle layout: 64-element atom columns of
// kTileRows x 128 B, 16-byte chunk c of row r at chunk position c ^ (r % 8).
__device__ __forceinline__ uint32_t sw128_offset(int row, int b)
{
    const int atom = b >> 7, o = b & 127;
    return atom * (kTileRows * 128) + row * 128 + ((((o >> 4) ^ (row & 7)) << 4) | (o & 15));
}

// Split C fp32 values into bf16 hi and lo and store this lane's slice of
// operand row `row` (elements lane*C .. lane*C + C - 1).
template <int C>
__device__ __forceinline__ void store_split(unsigned char* hi, unsigned char* lo, int row, int lane,
                                            const float (&v)[C])
{
    uint32_t hw[C / 2], lw[C / 2];
#pragma unroll
    for (int i = 0; i < C / 2; ++i) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]);
        const __nv_bfloat16 h1 = __float2bfloat16_rn(v[2 * i + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * i] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * i + 1] - __bfloat162float(h1));
        hw[i] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
        lw[i] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
    }
    const uint32_t off = sw128_offset(row, lane * C * 2);
    if constexpr (C == 4) {
        *reinterpret_cast<uint2*>(hi + off) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2*>(lo + off) = make_uint2(lw[0], lw[1]);
    } else {
        *reinterpret_cast<uint32_t*>(hi + off) = hw[0];
        *reinterpret_cast<uint32_t*>(lo + off) = lw[0];
    }
}

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 h)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(h.x)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h.y)) << 16);
}

// Split elements e0..e0+3 of operand row `row` into bf16 hi and lo (8 bytes each).
__device__ __forceinline__ void store_split4(unsigned char* hi, unsigned char* lo, int row, int e0, float4 v)
{
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
    const uint32_t off = sw128_offset(row, e0 * 2);
    *reinterpret_cast<uint2*>(hi + off) = make_uint2(bf2_bits(h01), bf2_bits(h23));
    *reinterpret_cast<uint2*>(lo + off) = make_uint2(bf2_bits(l01), bf2_bits(l23));
}

// Shared -> global through the TMA engine (both addresses 16-byte aligned, bytes a multiple of 16), one
// bulk async-group per commit; the issuing thread waits for the group's reads of shared memory (.read)
// before the buffer is written again, and for its completion before the CTA exits.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src_smem)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy writes to shared memory made visible to a later bulk copy's reads (each writing thread).
__device__ __forceinline__ void fence_smem_for_bulk() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 bytes global -> shared through the async-copy path (cached in L2 only).
__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// What a warp knows about one of its 32 rows (lane l describes row l).
template <typename IX>
struct RowMeta {
    int kind;  // 0 unused, 1 dense x, 2 bag of table t = k - 1 (or a pooled input row)
    int len;   // lookups in the bag
    IX start;  // first position of the bag in indices[]
    IX idx;    // the bag's index when len == 1 (read one tile ahead)
};

template <typename IX>
struct OffPair {
    IX s0, s1;
};

// Offsets of the bag behind warp row `lane` of tile `tile` (read two tiles ahead).
// IX is the index type: with int32 indices every position fits in 32 bits.
template <typename TI, int MODE, int NP>
__device__ __forceinline__ OffPair<TI> load_offsets(const FwdArgs& a, int64_t tile, int64_t num_tiles, int warp,
                                                    int lane)
{
    constexpr int S = kTileRows / NP;
    OffPair<TI> o{0, 0};
    const int rt = kWarp * warp + lane;
    const int k = rt % NP;
    if (MODE == kInteract || tile >= num_tiles || k == 0 || k > a.T) return o;
    const TI b = static_cast<TI>(tile * S + rt / NP);
    if (b >= a.B) return o;
    const TI bag = static_cast<TI>(k - 1) * static_cast<TI>(a.B) + b;
    const TI* off = static_cast<const TI*>(a.offsets);
    o.s0 = __ldg(off + bag);
    o.s1 = __ldg(off + bag + 1);
    return o;
}

// Bag range of the row; a one-lookup bag's index is read here (one tile ahead).
template <typename TI, int MODE, int NP>
__device__ __forceinline__ RowMeta<TI> stage_bag(const FwdArgs& a, int64_t tile, int64_t num_tiles, int warp,
                                                 int lane, OffPair<TI> o)
{
    constexpr int S = kTileRows / NP;
    RowMeta<TI> m{0, 0, 0, -1};
    const int rt = kWarp * warp + lane;
    const int k = rt % NP;
    if (tile >= num_tiles || k > a.T || tile * S + rt / NP >= a.B) return m;
    if (k == 0) {
        m.kind = 1;
        return m;
    }
    m.kind = 2;
    if (MODE == kInteract) {
        m.len = 1;
        return m;
    }
    if (o.s0 < 0 || o.s1 < o.s0 || o.s1 > static_cast<TI>(a.nnz)) {
        flag_status(a.status, DLRM_ERR_BAD_OFFSETS);  // treated as an empty bag
        return m;
    }
    m.len = static_cast<int>(o.s1 - o.s0);
    m.start = o.s0;
    if (m.len == 1) m.idx = __ldg(static_cast<const TI*>(a.indices) + o.s0);
    return m;
}

// Finish warp row rr from a value pooled in registers (C values per lane):
// stage x exactly, save the pooled bag when asked, split into the operands.
template <int D, int MODE, int NP>
__device__ __forceinline__ void finish_row(const FwdArgs& a, unsigned char* op_hi, unsigned char* op_lo,
                                           float* stage, int W, int64_t tile, int warp, int lane, int rr,
                                           const float (&v)[D / kWarp])
{
    constexpr int C = D / kWarp;
    constexpr int S = kTileRows / NP;
    const int rt = kWarp * warp + rr;
    const int k = rt % NP;
    if (k == 0) {  // x, exactly: straight to its output row in one-sample tiles, else to the staged row
        float* dst = S == 1 ? a.out + tile * W + lane * C : stage + (rt / NP) * W + lane * C;
#pragma unroll
        for (int c = 0; c < C; ++c) dst[c] = v[c];
    } else if (MODE == kFused && a.pooled_out != nullptr) {
        const int64_t b = tile * S + rt / NP;
        float* dst = a.pooled_out + (b * a.T + (k - 1)) * D + lane * C;
        if constexpr (C == 4)
            *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        else
            *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
    }
    store_split<C>(op_hi, op_lo, rt, lane, v);
}

// Pop up to G rows from a warp-uniform row mask; lane group g gets the g-th (or -1).
template <int G>
__device__ __forceinline__ int pop_rows(uint32_t& mask, int g)
{
    int mine = -1;
#pragma unroll
    for (int q = 0; q < G; ++q) {
        const int r = mask != 0 ? __ffs(mask) - 1 : -1;
        mask &= mask - 1;
        if (q == g) mine = r;
    }
    return mine;
}

// MULTI: bags of several lookups are pooled by the whole warp from one list of
// lookups (else one bag at a time, the rare case of a mostly one-hot batch).
// D = 64 without multi-lookup pooling fits 128 registers (no spills) and 56 KB of shared memory: 4 CTAs per
// SM instead of 3.
template <int D, typename TE, typename TI, int MODE, int NP, bool MULTI>
__global__ void __launch_bounds__(kThreads, (D == 64 && !MULTI) ? 4 : 3) forward_tc_kernel(const __grid_constant__ FwdArgs a, int64_t num_tiles)
{
    constexpr int C = D / kWarp;                 // columns per lane when pooling in registers
    constexpr int S = kTileRows / NP;            // samples per tile
    constexpr int SLICE = C * static_cast<int>(sizeof(TE));
    constexpr int REGION = kTileRows * 128;      // one 64-element atom column of an operand
    constexpr int F32_CHUNKS = D / 4;            // 16-byte chunks of an fp32 row: 32 or 16
    constexpr int BF_CHUNKS = D / 8;             // of a bf16 row: 16 or 8
    constexpr int F32_GROUPS = kWarp / F32_CHUNKS;  // fp32 rows split per pass: 1 or 2
    constexpr int BF_GROUPS = kWarp / BF_CHUNKS;    // bf16 rows per pass: 2 or 4
    constexpr int F32_SLOTS = kWarp / F32_GROUPS;   // rows each lane group handles: 32 or 16
    constexpr int BF_SLOTS = kWarp / BF_GROUPS;     // 16 or 8
    constexpr uint32_t F32_BYTES = D * 4;
    constexpr uint32_t TE_BYTES = D * sizeof(TE);
    using SliceT = Slice<SLICE>;
    // One-sample tiles store the output triangle through the TMA engine (a bulk copy from shared memory);
    // tiles of several short rows copy them out with coalesced stores of every thread.
    constexpr bool kBulkOut = S == 1;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int T = a.T, N = T + 1;
    const int W = D + N * (N - 1) / 2;
    const TcLayout L = make_tc_layout(D, S, W);
    unsigned char* op_hi = smem + L.hi;
    unsigned char* op_lo = smem + L.lo;  // = op_hi + D * 256: the four (D = 128) or two regions are contiguous
    float* stage = reinterpret_cast<float*>(smem + L.stage);
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot);
    const char** tab_base = reinterpret_cast<const char**>(smem + L.tables);
    int64_t* tab_rows = reinterpret_cast<int64_t*>(smem + L.tables + 8 * kMaxTablesTc);
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const bool mean = MODE == kFused && a.mean != 0;
    const bool save_pooled = MODE == kFused && a.pooled_out != nullptr;
    const int i0 = (kWarp * warp) % NP;  // first vector index of the warp's rows

    if (blockIdx.x == 0 && threadIdx.x == 0 && MODE != kInteract) {
        const int64_t first = load_idx<TI>(a.offsets, 0);
        const int64_t last = load_idx<TI>(a.offsets, static_cast<int64_t>(T) * a.B);
        if (first != 0 || last != a.nnz) flag_status(a.status, DLRM_ERR_BAD_OFFSETS);
    }
    for (int t = threadIdx.x; t < T; t += kThreads) {
        tab_base[t] = static_cast<const char*>(a.tables[t]);
        tab_rows[t] = a.num_rows[t];
    }
    if (threadIdx.x == 0) {
        mbar_init(mma_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int64_t G = gridDim.x;
    uint32_t mma_phase = 0;
    bool timed_out = false, mma_pending = false;
    int64_t tile = blockIdx.x;
    OffPair<TI> o_next = load_offsets<TI, MODE, NP>(a, tile + G, num_tiles, warp, lane);
    RowMeta<TI> m = stage_bag<TI, MODE, NP>(a, tile, num_tiles, warp, lane,
                                            load_offsets<TI, MODE, NP>(a, tile, num_tiles, warp, lane));
    // One-sample tiles (NP = 128) issue the next tile's rows as soon as this tile's MMAs have read the
    // operands, so they travel during the epilogue and the output stores (a long phase at N > 64); the next
    // iteration then only takes the masks saved here.  (The loop top below stays as it is for every tile
    // shape: for NP < 128 `pre` is a compile-time false and that code is unchanged.)
    uint32_t early_f32 = 0, early_bf = 0, early_empty = 0;
    bool early = false;
    auto issue_early = [&](int64_t tl, const RowMeta<TI>& mm) {
        const int rt = kWarp * warp + lane;
        const int k = rt % NP;
        const int64_t b = tl * S + rt / NP;
        const char* src = nullptr;
        uint32_t bytes = 0;
        if (mm.kind == 1) {
            src = reinterpret_cast<const char*>(a.dense + b * D);
            bytes = F32_BYTES;
        } else if (mm.kind == 2) {
            if (MODE == kInteract) {
                src = reinterpret_cast<const char*>(a.pooled_in + (b * T + (k - 1)) * D);
                bytes = F32_BYTES;
            } else if (mm.len == 1) {
                if (mm.idx >= 0 && mm.idx < tab_rows[k - 1]) {
                    src = tab_base[k - 1] + static_cast<uint64_t>(mm.idx) * TE_BYTES;
                    bytes = TE_BYTES;
                } else {
                    flag_status(a.status, DLRM_ERR_INDEX_OOB);  // contributes zero, still counts in L
                }
            }
        }
        early_f32 = __ballot_sync(kFull, bytes != 0 && bytes == F32_BYTES);
        early_bf = __ballot_sync(kFull, bytes != 0 && bytes != F32_BYTES);
        early_empty = __ballot_sync(kFull, mm.kind == 2 && bytes == 0 && (MODE == kInteract || mm.len <= 1));
        const int g32 = lane / F32_CHUNKS, c32 = lane % F32_CHUNKS;
        unsigned char* const raw_lane = op_hi + (c32 >> 3) * REGION + (c32 & 7) * 16 + (kWarp * warp + g32 * F32_SLOTS) * 128;
#pragma unroll
        for (int q = 0; q < F32_SLOTS; ++q) {
            const int r = g32 * F32_SLOTS + q;
            const char* p = reinterpret_cast<const char*>(shfl64(reinterpret_cast<int64_t>(src), r));
            if ((early_f32 >> r) & 1u) cp_async16(raw_lane + q * 128, p + c32 * 16);
        }
        if (sizeof(TE) == 2) {
            const int gb = lane / BF_CHUNKS, cb = lane % BF_CHUNKS;
            unsigned char* const hi_lane = op_hi + (cb >> 3) * REGION;
#pragma unroll
            for (int q = 0; q < BF_SLOTS; ++q) {
                const int r = gb * BF_SLOTS + q;
                const int row = kWarp * warp + r;
                const char* p = reinterpret_cast<const char*>(shfl64(reinterpret_cast<int64_t>(src), r));
                if ((early_bf >> r) & 1u) cp_async16(hi_lane + row * 128 + (((cb & 7) ^ (r & 7)) << 4), p + cb * 16);
            }
        }
        cp_async_commit();
        early = true;
    };

    for (; tile < num_tiles; tile += G) {
        const bool pre = NP == kTileRows && early;  // this tile's rows were issued during the last epilogue
        early = false;
        // ---- every single-row source of the warp in flight at once, straight into the operand lines ----
        // An fp32 row lands unswizzled in the four (D = 128) or two 128-byte lines its hi / lo halves
        // will occupy and is split there in place; a bf16 row lands at its final, swizzled hi position
        // (lo = 0).  The warp moves F32_GROUPS (bf16: BF_GROUPS) rows per instruction, 16 bytes a lane.
        const int rt = kWarp * warp + lane;
        const int k = rt % NP;
        const int64_t b = tile * S + rt / NP;
        const char* src = nullptr;
        uint32_t bytes = 0;
        if (pre) {
        } else if (m.kind == 1) {
            src = reinterpret_cast<const char*>(a.dense + b * D);
            bytes = F32_BYTES;
        } else if (m.kind == 2) {
            if (MODE == kInteract) {
                src = reinterpret_cast<const char*>(a.pooled_in + (b * T + (k - 1)) * D);
                bytes = F32_BYTES;
            } else if (m.len == 1) {
                if (m.idx >= 0 && m.idx < tab_rows[k - 1]) {
                    src = tab_base[k - 1] + static_cast<uint64_t>(m.idx) * TE_BYTES;
                    bytes = TE_BYTES;
                } else {
                    flag_status(a.status, DLRM_ERR_INDEX_OOB);  // contributes zero, still counts in L
                }
            }
        }
        const bool f32row = bytes == F32_BYTES;
        const uint32_t conv_f32 = pre ? early_f32 : __ballot_sync(kFull, bytes != 0 && f32row);
        const uint32_t conv_bf = pre ? early_bf : __ballot_sync(kFull, bytes != 0 && !f32row);
        const uint32_t empty =
            pre ? early_empty : __ballot_sync(kFull, m.kind == 2 && bytes == 0 && (MODE == kInteract || m.len <= 1));
        // lane group g (F32_CHUNKS lanes, one 16-byte chunk each) moves rows g * SLOTS .. g * SLOTS + SLOTS - 1
        const int g32 = lane / F32_CHUNKS, c32 = lane % F32_CHUNKS;
        unsigned char* const raw_lane = op_hi + (c32 >> 3) * REGION + (c32 & 7) * 16 + (kWarp * warp + g32 * F32_SLOTS) * 128;
#pragma unroll
        for (int q = 0; q < F32_SLOTS; ++q) {
            const int r = g32 * F32_SLOTS + q;
            const char* p = reinterpret_cast<const char*>(shfl64(reinterpret_cast<int64_t>(src), r));
            if (!pre && ((conv_f32 >> r) & 1u)) cp_async16(raw_lane + q * 128, p + c32 * 16);
        }
        if (sizeof(TE) == 2) {
            const int gb = lane / BF_CHUNKS, cb = lane % BF_CHUNKS;
            unsigned char* const hi_lane = op_hi + (cb >> 3) * REGION;
#pragma unroll
            for (int q = 0; q < BF_SLOTS; ++q) {
                const int r = gb * BF_SLOTS + q;
                const int row = kWarp * warp + r;
                const char* p = reinterpret_cast<const char*>(shfl64(reinterpret_cast<int64_t>(src), r));
                if (!pre && ((conv_bf >> r) & 1u))  // straight to the swizzled hi position: a bf16 row is its own hi, lo = 0
                    cp_async16(hi_lane + row * 128 + (((cb & 7) ^ (r & 7)) << 4), p + cb * 16);
            }
        }
        if (!pre) cp_async_commit();

        // ---- the next tiles' metadata while these rows travel ----
        const RowMeta<TI> m_next = stage_bag<TI, MODE, NP>(a, tile + G, num_tiles, warp, lane, o_next);
        o_next = load_offsets<TI, MODE, NP>(a, tile + 2 * G, num_tiles, warp, lane);

        // ---- bags of several lookups: the warp's lookups as one list, 16 rows in flight, each summed
        //      in lookup order in registers; a finished sum goes to its row's lines as an fp32 row ----
        uint32_t multi = 0, pooled_rows = 0, zero_rows = 0;
        if (MODE == kFused && MULTI) multi = __ballot_sync(kFull, m.len > 1);
        if (MULTI && multi != 0) {
            using Slice4 = Slice<4 * static_cast<int>(sizeof(TE))>;
            const bool lane_on = lane < F32_CHUNKS;  // lane l sums elements 4l .. 4l + 3
            const int lenm = ((multi >> lane) & 1u) ? m.len : 0;
            int incl = lenm;
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            const int total = __shfl_sync(kFull, incl, kWarp - 1);
            uint32_t started = 0;  // rows that received a valid lookup
            int cur = -1;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            auto store_cur = [&]() {
                if (cur >= 0 && ((started >> cur) & 1u) && lane_on)
                    *reinterpret_cast<float4*>(op_hi + (lane >> 3) * REGION + (kWarp * warp + cur) * 128 + (lane & 7) * 16) = acc;
            };
            for (int q0 = 0; q0 < total; q0 += kWarp) {
                // lane l resolves lookup q = q0 + l: its row is the number of rows whose list ends at or before q
                const int q = q0 + lane;
                int r = 0;
#pragma unroll
                for (int bit = 16; bit > 0; bit >>= 1) {
                    const int e = __shfl_sync(kFull, incl, r + bit - 1);
                    if (e <= q) r += bit;
                }
                const int rs = r & (kWarp - 1);
                const int beg = __shfl_sync(kFull, incl - lenm, rs);
                const int64_t st = static_cast<int64_t>(__shfl_sync(kFull, static_cast<long long>(m.start), rs));
                const char* src = nullptr;
                if (q < total) {
                    const int t_r = (kWarp * warp + r) % NP - 1;
                    const int64_t idx = load_idx<TI>(a.indices, st + (q - beg));
                    if (idx >= 0 && idx < tab_rows[t_r])
                        src = tab_base[t_r] + static_cast<uint64_t>(idx) * TE_BYTES;
                    else
                        flag_status(a.status, DLRM_ERR_INDEX_OOB);  // contributes zero, still counts in L
                }
                const uint32_t vmask = __ballot_sync(kFull, src != nullptr);
#pragma unroll 1
                for (int h = 0; h < kWarp; h += 16) {
                    if (q0 + h >= total) break;
                    Slice4 raw[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const char* p = reinterpret_cast<const char*>(shfl64(reinterpret_cast<int64_t>(src), h + u));
                        if (p != nullptr && lane_on) raw[u].load(p, lane);
                    }
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        if (q0 + h + u >= total) break;
                        const int ru = __shfl_sync(kFull, r, h + u);
                        if (ru != cur) {
                            store_cur();
                            cur = ru;
                        }
                        if ((vmask >> (h + u)) & 1u) {
                            float f[4];
                            widen<4, TE>(raw[u], f);
                            if ((started >> cur) & 1u) {  // packed adds: each lane an fp32 add, rounded once
                                const float2 a01 = __fadd2_rn(make_float2(acc.x, acc.y), make_float2(f[0], f[1]));
                                const float2 a23 = __fadd2_rn(make_float2(acc.z, acc.w), make_float2(f[2], f[3]));
                                acc = make_float4(a01.x, a01.y, a23.x, a23.y);
                            } else {  // a sum starts from its first term
                                acc = make_float4(f[0], f[1], f[2], f[3]);
                                started |= 1u << cur;
                            }
                        }
                    }
                }
            }
            store_cur();
            pooled_rows = started;
            zero_rows = multi & ~started;  // every lookup out of range: the bag pools to zero
        }

        // ---- empty bags (or bags whose every index is out of range) pool to zero ----
        {
            uint32_t mask = empty | zero_rows;
            const int g = lane / F32_CHUNKS, gl = lane % F32_CHUNKS;
            while (mask != 0) {
                const int r = pop_rows<F32_GROUPS>(mask, g);
                if (r < 0) continue;
                const int row = kWarp * warp + r;
                *reinterpret_cast<uint4*>(op_hi + (gl >> 3) * REGION + row * 128 + (gl & 7) * 16) = make_uint4(0, 0, 0, 0);
                if (save_pooled) {
                    const int64_t br = tile * S + row / NP;
                    *reinterpret_cast<float4*>(a.pooled_out + (br * T + (row % NP - 1)) * D + gl * 4) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }

        // ---- rows of longer bags, one at a time: 8 lookups in flight, summed in lookup order ----
        if (MODE == kFused && !MULTI) {
            uint32_t multi = __ballot_sync(kFull, m.len > 1);
            while (multi != 0) {
                const int rr = __ffs(multi) - 1;
                multi &= multi - 1;
                const int Lr = __shfl_sync(kFull, m.len, rr);
                const int64_t st_r = static_cast<int64_t>(__shfl_sync(kFull, static_cast<long long>(m.start), rr));
                const int t_r = (kWarp * warp + rr) % NP - 1;
                const char* base_r = tab_base[t_r];
                const int64_t V_r = tab_rows[t_r];
                float acc[C];
#pragma unroll
                for (int c = 0; c < C; ++c) acc[c] = 0.0f;
                bool started = false;
                for (int p0 = 0; p0 < Lr; p0 += kWarp) {
                    const int n = min(kWarp, Lr - p0);
                    int64_t my_idx = -1;
                    if (lane < n) {
                        my_idx = load_idx<TI>(a.indices, st_r + p0 + lane);
                        if (my_idx < 0 || my_idx >= V_r) {
                            flag_status(a.status, DLRM_ERR_INDEX_OOB);  // contributes zero, still counts in L
                            my_idx = -1;
                        }
                    }
                    for (int u0 = 0; u0 < n; u0 += 8) {
                        SliceT raw[8];
                        bool ok[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int64_t idx = shfl64(my_idx, (u0 + u) & (kWarp - 1));
                            ok[u] = u0 + u < n && idx >= 0;
                            if (ok[u]) raw[u].load(base_r + idx * static_cast<int64_t>(TE_BYTES), lane);
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            if (!ok[u]) continue;
                            float f[C];
                            widen<C, TE>(raw[u], f);
#pragma unroll
                            for (int c = 0; c < C; ++c) acc[c] = started ? acc[c] + f[c] : f[c];
                            started = true;
                        }
                    }
                }
                float v[C];
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    float x = started ? acc[c] : 0.0f;
                    if (mean && started) x = __fdiv_rn(x, static_cast<float>(Lr));
                    v[c] = x;
                }
                finish_row<D, MODE, NP>(a, op_hi, op_lo, stage, W, tile, warp, lane, rr, v);
            }
        }

        // ---- the rows have landed: split fp32 rows into hi / lo in place; bf16 rows get lo = 0 ----
        cp_async_wait_all();
        __syncwarp();
        {
            {
                // lane group g32 splits rows g32 * F32_SLOTS + q, four at a time: loads first, then the math.
                // A pooled bag of a mean-pooled table is divided by its length here.
                const uint32_t conv_rows = conv_f32 | pooled_rows;
                const bool x_warp = i0 == 0 && (conv_f32 & 1u);  // row 0 of this warp is a dense vector x
                const bool scale = mean && pooled_rows != 0;
#pragma unroll
                for (int q0 = 0; q0 < F32_SLOTS; q0 += 4) {
                    float4 v[4];
                    int Lq[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        Lq[q] = scale ? __shfl_sync(kFull, m.len, g32 * F32_SLOTS + q0 + q) : 1;
                        if ((conv_rows >> (g32 * F32_SLOTS + q0 + q)) & 1u)
                            v[q] = *reinterpret_cast<const float4*>(raw_lane + (q0 + q) * 128);
                    }
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = g32 * F32_SLOTS + q0 + q;
                        if (!((conv_rows >> r) & 1u)) continue;
                        const int row = kWarp * warp + r;
                        if (scale && ((pooled_rows >> r) & 1u)) {
                            const float fl = static_cast<float>(Lq[q]);
                            v[q] = make_float4(__fdiv_rn(v[q].x, fl), __fdiv_rn(v[q].y, fl), __fdiv_rn(v[q].z, fl),
                                               __fdiv_rn(v[q].w, fl));
                        }
                        if (q0 + q == 0 && g32 == 0 && x_warp) {  // x, exactly (see the output stores)
                            float* dst = kBulkOut ? a.out + tile * W + c32 * 4 : stage + (row / NP) * W + c32 * 4;
                            dst[0] = v[q].x;
                            dst[1] = v[q].y;
                            dst[2] = v[q].z;
                            dst[3] = v[q].w;
                        } else if (save_pooled) {
                            const int64_t br = tile * S + row / NP;
                            *reinterpret_cast<float4*>(a.pooled_out + (br * T + (row % NP - 1)) * D + c32 * 4) = v[q];
                        }
                        store_split4(op_hi, op_lo, row, c32 * 4, v[q]);
                    }
                }
            }
            if (sizeof(TE) == 2 && MODE == kFused) {
                uint32_t mask = conv_bf;
                const int g = lane / BF_CHUNKS, gl = lane % BF_CHUNKS;
                const int line_off = (gl >> 3) * REGION + (gl & 7) * 16;
                while (mask != 0) {
                    const int r = pop_rows<BF_GROUPS>(mask, g);
                    if (r < 0) continue;
                    const int row = kWarp * warp + r;
                    const int sw_off = (gl >> 3) * REGION + row * 128 + (((gl & 7) ^ (row & 7)) << 4);
                    *reinterpret_cast<uint4*>(op_lo + line_off + row * 128) = make_uint4(0, 0, 0, 0);
                    if (save_pooled) {
                        const int64_t br = tile * S + row / NP;
                        const uint4 h = *reinterpret_cast<const uint4*>(op_hi + sw_off);
                        float f[8];
                        bf16x8_to_f32(h, f);
                        float4* dst = reinterpret_cast<float4*>(a.pooled_out + (br * T + (row % NP - 1)) * D + gl * 8);
                        dst[0] = make_float4(f[0], f[1], f[2], f[3]);
                        dst[1] = make_float4(f[4], f[5], f[6], f[7]);
                    }
                }
            }
        }

        // ---- the Gram of the tile on the tensor cores ----
        tc::fence_smem_for_mma();
        __syncthreads();
        if (threadIdx.x == 0) {
            tc::fence_after_sync();
            const uint32_t a_hi = smem_addr(op_hi), a_lo = smem_addr(op_lo);
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kTileRows, kTileRows);
            constexpr int KS = D / 16;  // MMAs of K = 16 per product
#pragma unroll 1
            for (int it = 0; it < 3 * KS; ++it) {  // hi*hi, hi*lo, lo*hi
                const int pass = it / KS, ks = it - pass * KS;
                const uint32_t off = (ks >> 2) * REGION + (ks & 3) * 32;
                const uint32_t A = (pass == 2 ? a_lo : a_hi) + off;
                const uint32_t B = (pass == 1 ? a_lo : a_hi) + off;
                tc::mma_bf16(tmem, tc::desc_kmajor_sw128(A), tc::desc_kmajor_sw128(B), idesc, it != 0);
            }
            tc::commit(mma_bar);
            if constexpr (kBulkOut) bulk_wait_read();  // the last tile's output stores have read the staging area
        }
        mma_pending = true;
        m = m_next;

        const bool done = mbar_wait_bounded(mma_bar, mma_phase);
        if (__syncthreads_or(!done)) {
            timed_out = true;
            break;
        }
        mma_pending = false;
        mma_phase ^= 1;
        tc::fence_after_sync();
        if constexpr (NP == kTileRows) {
            if (tile + G < num_tiles) issue_early(tile + G, m);  // m already holds the next tile's rows
        }

        // ---- epilogue: this warp's rows of its sample's diagonal block ----
        {
            const int sw = (kWarp * warp) / NP;      // sample slot of the warp
            const int i = i0 + lane;
            const int64_t bw = tile * S + sw;
            if (bw < a.B && i0 < N) {
                // one-sample tiles: the triangle starts at the same 16-byte residue as its place in out
                const int sh =
                    kBulkOut ? static_cast<int>((reinterpret_cast<uintptr_t>(a.out + bw * W + D) >> 2) & 3u) : 0;
                float* st = kBulkOut ? stage + sh - D : stage + sw * W;
                const int base_i = D + i * N - i * (i + 1) / 2 - i - 1;  // out position of (i, j) is base_i + j
                for (int cb = i0 / kWarp; cb * kWarp < N; ++cb) {
                    uint32_t z[32];
                    tc::tmem_ld_32x32b_x32(tmem + ((static_cast<uint32_t>(kWarp * warp)) << 16) +
                                               static_cast<uint32_t>(sw * NP + cb * kWarp),
                                           z);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int j = cb * kWarp + jj;
                        if (j > i && j < N) st[base_i + j] = __uint_as_float(z[jj]);
                    }
                }
            }
        }
        if constexpr (kBulkOut) fence_smem_for_bulk();  // the staged triangle, written by every thread, to the TMA engine
        tc::fence_before_sync();
        __syncthreads();

        if constexpr (kBulkOut) {
            // ---- one-sample tile (a long triangle): its 16-byte aligned body by one bulk copy from thread 0,
            //      which also waits for it; a head and a tail of at most 3 floats by plain stores (x went out
            //      in the split) ----
            if (tile < a.B) {
                const int Wt = W - D;
                float* o = a.out + tile * W + D;
                const int sh = static_cast<int>((reinterpret_cast<uintptr_t>(o) >> 2) & 3u);
                const int head = min((4 - sh) & 3, Wt);
                const int body = (Wt - head) & ~3;
                const float* st = stage + sh;
                if (threadIdx.x == 0) {
                    if (body > 0) bulk_s2g(o + head, st + head, static_cast<uint32_t>(body) * 4u);
                    bulk_commit();
                } else if (warp == 1 && lane < 6) {  // lanes 0..2: the head, 3..5: the tail
                    const int t = head + body + (lane - 3);
                    if (lane < 3 && lane < head) o[lane] = st[lane];
                    if (lane >= 3 && t < Wt) o[t] = st[t];
                }
            }
        } else {
            // ---- the tile's output rows, coalesced ----
            const int64_t b0 = tile * S;
            const int ns = static_cast<int>(min(static_cast<int64_t>(S), a.B - b0));
            float* o = a.out + b0 * W;
            for (int e = threadIdx.x; e < ns * W; e += kThreads) o[e] = stage[e];
        }
        __syncthreads();  // operands free for the next tile (the staging area once the bulk reads are done)
    }

    if constexpr (kBulkOut) {
        if (threadIdx.x == 0) bulk_wait_done();  // the output stores are complete before the CTA exits
    }
    if (timed_out) {
        if (threadIdx.x == 0) flag_status(a.status, DLRM_ERR_TIMEOUT);
        // let copies and an MMA still in flight finish (bounded) before shared memory and TMEM are released
        if (mma_pending) mbar_wait_bounded(mma_bar, mma_phase);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
constexpr int kMaxSmem = 227 * 1024;
constexpr int kSmemPerSm = 228 * 1024;

template <int D, typename TE, typename TI, int MODE, int NP, bool MULTI>
dlrm_status launch_tc(const FwdArgs& a, cudaStream_t stream)
{
    constexpr int S = kTileRows / NP;
    const int N = a.T + 1;
    const int W = D + N * (N - 1) / 2;
    const TcLayout L = make_tc_layout(D, S, W);
    int smem = L.bytes + 1024;  // + alignment of the operands to 1024 bytes
    if (smem < kMinSmemPerCta) smem = kMinSmemPerCta;
    if (smem > kMaxSmem) return DLRM_ERR_UNSUPPORTED;
    auto kern = forward_tc_kernel<D, TE, TI, MODE, NP, MULTI>;
    // Function attributes belong to the current device's context: set them on every launch (a cheap host
    // call), so that every device, and a context made again after a reset, gets them.
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return DLRM_ERR_CUDA;
    const int regs = kernel_registers(reinterpret_cast<const void*>(kern));
    if (regs <= 0) return DLRM_ERR_CUDA;
    // CTAs per SM: shared memory (1 KB of it reserved per CTA), registers, TMEM
    int per_sm = kSmemPerSm / (smem + 1024);
    const int by_regs = 65536 / (round_up(regs, 8) * kThreads);
    if (by_regs < per_sm) per_sm = by_regs;
    if (per_sm > kMaxCtasPerSm) per_sm = kMaxCtasPerSm;
    const int sms = sm_count();
    if (per_sm < 1 || sms < 1) return DLRM_ERR_UNSUPPORTED;
    const int64_t tiles = (a.B + S - 1) / S;
    const int64_t grid = tiles < static_cast<int64_t>(sms) * per_sm ? tiles : static_cast<int64_t>(sms) * per_sm;
    kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a, tiles);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

template <int D, typename TE, typename TI, int MODE, bool MULTI>
dlrm_status dispatch_np(const FwdArgs& a, cudaStream_t s)
{
    const int N = a.T + 1;
    if (N <= 32) return launch_tc<D, TE, TI, MODE, 32, MULTI>(a, s);
    if (N <= 64) return launch_tc<D, TE, TI, MODE, 64, MULTI>(a, s);
    return launch_tc<D, TE, TI, MODE, 128, MULTI>(a, s);
}

// Bags average more than 1.25 lookups: the multi-lookup variant.
inline bool multi_hot(const FwdArgs& a) { return 4 * a.nnz > 5 * static_cast<int64_t>(a.T) * a.B; }

template <int D, typename TE, typename TI>
dlrm_status dispatch_fused(const FwdArgs& a, cudaStream_t s)
{
    return multi_hot(a) ? dispatch_np<D, TE, TI, kFused, true>(a, s) : dispatch_np<D, TE, TI, kFused, false>(a, s);
}

template <int D>
dlrm_status dispatch_tc(int mode, const FwdArgs& a, int dtype, int index_type, cudaStream_t s)
{
    if (mode == kInteract) return dispatch_np<D, float, int32_t, kInteract, false>(a, s);
    if (dtype == DLRM_F32)
        return index_type == DLRM_I32 ? dispatch_fused<D, float, int32_t>(a, s) : dispatch_fused<D, float, int64_t>(a, s);
    return index_type == DLRM_I32 ? dispatch_fused<D, __nv_bfloat16, int32_t>(a, s)
                                  : dispatch_fused<D, __nv_bfloat16, int64_t>(a, s);
}

}  // namespace

bool forward_tc_supported(int mode, int dim, int num_tables, int64_t batch, int64_t nnz)
{
    if (!((mode == kFused || mode == kInteract) && (dim == 64 || dim == 128) && num_tables + 1 <= kTileRows))
        return false;
    // bags averaging more than 16 lookups are pooled faster by the register-pooling kernel,
    // whose half-warps read two rows per instruction
    return mode == kInteract || nnz <= 16 * static_cast<int64_t>(num_tables) * batch;
}

dlrm_status launch_forward_tc(int mode, const FwdArgs& a, int dim, int dtype, int index_type, cudaStream_t s)
{
    switch (dim) {
        case 64: return dispatch_tc<64>(mode, a, dtype, index_type, s);
        case 128: return dispatch_tc<128>(mode, a, dtype, index_type, s);
        default: return DLRM_ERR_UNSUPPORTED;
    }
}

}  // namespace dlrm
