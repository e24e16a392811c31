// mlp.cu -- the dense layers around the sparse path: the bottom MLP, the top
// MLP and the sigmoid output with its binary cross-entropy loss, forward and
// backward with plain SGD on their weights ("DLRM", robocikowo.com, "Forward
// pass" steps (1) and (4), the bottom-MLP and top-MLP paragraphs: FC layers
// with ReLU, a sigmoid output; the hardware paragraph: the MLPs are ordinary
// GEMMs on the tensor cores).
//
// GEMM.  C[M x N] = A[M x K] * B[N x K]^T with both operands K-major (a row of
// A or B holds its K values contiguously), on the tcgen05 tensor cores.  Each
// fp32 operand is first split once into bf16 hi = bf16(v) and lo = bf16(v - hi)
// arrays (K padded to a multiple of 8).  A CTA of 128 threads owns a 128 x 128
// tile of C: one thread issues cp.async.bulk.tensor loads of 64-wide K slices
// (128-byte swizzle, A hi / lo and B hi / lo, 64 KB) into a ring of 3 stages,
// another issues hi*hi^T + hi*lo^T + lo*hi^T (12 MMAs of 128 x 128 x 16 per
// slice) into a 128-column fp32 accumulator in TMEM and frees each stage by
// commit.  The dropped lo*lo term and the rounding of lo stay below 2^-16
// relative to sum |a_k b_k|.  Epilogue: all four warps read their 32 rows of the
// accumulator, add the bias and apply ReLU (or write a split-K partial), and
// store through a transpose in shared memory so that stores are row-contiguous.
//
// Backward of y = act(x W^T + b) from dy: dz = dy * [y > 0] (ReLU) or dy;
// dx = dz W; dW = dz^T x; db = sum over the batch of dz.  dz (the mask applied
// while it is split), x and W are each split once, row by row; the transposed
// operands (W in dx, dz and x in dW) are the same arrays read MN-major by the
// tensor cores, so nothing is transposed in memory.  dW is split over the batch
// into partial sums that the update kernel adds in a fixed order (bitwise
// reproducible) before W -= lr dW, b -= lr db.
//
// Head.  The last top layer maps to one logit: a warp per sample computes
// z = h . w + b, p = sigmoid(z), the sample's BCE term max(z, 0) - z y +
// log(1 + exp(-|z|)) and dz = (p - y) / M, writes dh = dz w, and the block adds
// its samples' dz h, dz and loss terms in a fixed order; a reduce kernel sums the
// blocks' partials in order, writes the mean loss and applies SGD to w and b.
#include <cuda.h>
#include <cuda_bf16.h>

#include <string.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dlrm {
namespace {

constexpr int kEpiWarps = 4;                    // warps 2-5: the epilogue, one per quarter of the TMEM lanes
constexpr int kGThreads = (2 + kEpiWarps) * 32;  // warp 0: TMA producer, warp 1: MMA issuer
constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kStages = 3;
constexpr int kTile = kBM * kBK * 2;        // one bf16 operand tile, 16 KB (kBM == kBN)
constexpr int kStage = 4 * kTile;           // A hi, A lo, B hi, B lo: 64 KB
constexpr int kEpiBytes = kEpiWarps * 32 * 33 * 4;  // the epilogue's transposes
constexpr int kGemmSmem = kStages * kStage + 1024 + 128 + kEpiBytes;
constexpr uint32_t kFull = 0xffffffffu;

// An operand is K-major (bf16 [rows x Kp] with the K values of a row contiguous; box 64 K x 128 rows) or
// MN-major (bf16 [K x MNp] with the M (or N) values of one k contiguous; box 64 M x 64 K, two boxes per
// 128-wide tile).  Both land as 16 KB per operand and stage in the 128-byte swizzle layout.
struct GemmArgs {
    CUtensorMap a_hi, a_lo, b_hi, b_lo;
    int a_mn, b_mn;                      // MN-major A / B
    const float* bias;                   // optional, N values
    float* c;
    int64_t ldc;
    int64_t M, N, K;
    int64_t splits;        // split-K: tiles z = 0 .. splits - 1 of each output tile
    int64_t k_per_split;   // reduction range of split z: [z * k_per_split, min(K, (z + 1) * k_per_split))
    int64_t split_stride;  // elements between the C partials of consecutive splits
    int relu;
    int32_t* status;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory matrix descriptor of an MN-major bf16 operand in the 128-byte swizzle layout: a 128-B row
// holds 64 consecutive M (or N) values of one k, consecutive k are consecutive rows, 8-row groups 1024 B
// apart (stride byte offset), the next 64 M (or N) values kMnBlock bytes later (leading byte offset).
// Moving the start by 2048 B selects the next 16 of K.
constexpr uint32_t kMnBlock = kBK * 128;  // one 64 x 64 box: 8 KB
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4)  // start address
           | (static_cast<uint64_t>(kMnBlock >> 4) << 16)   // leading byte offset: next 64 of M (or N)
           | (static_cast<uint64_t>(1024 >> 4) << 32)       // stride byte offset: next 8 rows of K
           | (static_cast<uint64_t>(1) << 46)               // descriptor version of tcgen05
           | (static_cast<uint64_t>(2) << 61);              // 128-byte swizzle
}

// Transpose bits of the kind::f16 instruction descriptor: A (bit 15), B (bit 16) MN-major.
constexpr uint32_t kIdescAMn = 1u << 15, kIdescBMn = 1u << 16;

// One CTA per SM walks tiles blockIdx.x, + gridDim.x, ... (M fastest, so CTAs running at once share B
// tiles in L2).  Warp 0 (one thread) loads slices into the ring, warp 1 (one thread) issues the MMAs of a
// tile into one of two TMEM accumulators, warps 2-5 drain the other accumulator: tile i's epilogue runs
// beside tile i + 1's MMAs.
__global__ void __launch_bounds__(kGThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmArgs g)
{
    extern __shared__ unsigned char gsm_raw[];
    unsigned char* sm = gsm_raw + ((1024u - (smem_addr(gsm_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kStages * kStage);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;  // [2] the MMAs of the accumulator's tile completed
    uint64_t* acc_empty = acc_full + 2;    // [2] the epilogue has read the accumulator out
    uint64_t* done = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    float* epi = reinterpret_cast<float*>(sm + kStages * kStage + 128);  // 4 x 32 x 33 floats
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t mt = (g.M + kBM - 1) / kBM, nt = (g.N + kBN - 1) / kBN;
    const int64_t tiles = mt * nt * g.splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], kEpiWarps);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, 2 * kBN);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    auto tile = [&](int s, int which) { return sm + s * kStage + which * kTile; };
    // tile t: rows m0, columns n0, reduction range [kb, ke) in nk slices
    struct Tile {
        int64_t m0, n0, z, kb;
        int nk;
    };
    auto tile_of = [&](int64_t t) {
        Tile r;
        r.z = t / (mt * nt);
        const int64_t rem = t - r.z * mt * nt;
        r.m0 = (rem % mt) * kBM;
        r.n0 = (rem / mt) * kBN;
        r.kb = r.z * g.k_per_split;
        const int64_t ke = min(g.K, r.kb + g.k_per_split);
        r.nk = ke > r.kb ? static_cast<int>((ke - r.kb + kBK - 1) / kBK) : 0;
        return r;
    };

    bool ok = true;
    if (warp == 0 && lane == 0) {
        // producer: the q-th slice of this CTA goes to stage q % kStages once the MMAs of slice q - kStages
        // have read it
        uint32_t q = 0;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            const Tile tl = tile_of(t);
            for (int i = 0; i < tl.nk && ok; ++i, ++q) {
                const int s = static_cast<int>(q % kStages);
                if (q >= kStages) ok = mbar_wait_bounded(&empty[s], ((q / kStages) - 1) & 1);
                if (!ok) break;
                mbar_arrive_expect_tx(&full[s], kStage);
                const int k = static_cast<int>(tl.kb + static_cast<int64_t>(i) * kBK);
                auto load = [&](int which, const CUtensorMap* map, int mn_major, int64_t row0) {
                    if (mn_major) {  // two 64 x 64 boxes: M (or N) values row0 .. +63, then +64 .. +127
                        tma_load_2d(tile(s, which), map, static_cast<int>(row0), k, &full[s]);
                        tma_load_2d(tile(s, which) + kMnBlock, map, static_cast<int>(row0) + 64, k, &full[s]);
                    } else {
                        tma_load_2d(tile(s, which), map, k, static_cast<int>(row0), &full[s]);
                    }
                };
                load(0, &g.a_hi, g.a_mn, tl.m0);
                load(1, &g.a_lo, g.a_mn, tl.m0);
                load(2, &g.b_hi, g.b_mn, tl.n0);
                load(3, &g.b_lo, g.b_mn, tl.n0);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: per slice hi*hi, hi*lo, lo*hi over 4 steps of K = 16, the stage released on commit;
        // per tile the accumulator j % 2, once the epilogue has drained it (tile j - 2)
        const uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN) | (g.a_mn ? kIdescAMn : 0u) | (g.b_mn ? kIdescBMn : 0u);
        // the next 16 of K: 32 B along a K-major row, 2048 B (16 rows) down an MN-major tile
        const uint32_t a_step = g.a_mn ? 2048u : 32u, b_step = g.b_mn ? 2048u : 32u;
        uint32_t q = 0, j = 0;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++j) {
            const Tile tl = tile_of(t);
            const uint32_t acc = j & 1u;
            if (j >= 2) ok = mbar_wait_bounded(&acc_empty[acc], ((j / 2) - 1) & 1);
            if (!ok) break;
            tc::fence_after_sync();
            const uint32_t d = tmem + acc * kBN;
            for (int i = 0; i < tl.nk && ok; ++i, ++q) {
                const int s = static_cast<int>(q % kStages);
                ok = mbar_wait_bounded(&full[s], (q / kStages) & 1);
                if (!ok) break;
                tc::fence_after_sync();
                const uint32_t ah = smem_addr(tile(s, 0)), al = smem_addr(tile(s, 1));
                const uint32_t bh = smem_addr(tile(s, 2)), bl = smem_addr(tile(s, 3));
#pragma unroll
                for (int it = 0; it < 12; ++it) {
                    const int pass = it / 4, ks = it % 4;
                    const uint32_t A = (pass == 2 ? al : ah) + ks * a_step;
                    const uint32_t B = (pass == 1 ? bl : bh) + ks * b_step;
                    const uint64_t da = g.a_mn ? desc_mnmajor_sw128(A) : tc::desc_kmajor_sw128(A);
                    const uint64_t db = g.b_mn ? desc_mnmajor_sw128(B) : tc::desc_kmajor_sw128(B);
                    tc::mma_bf16(d, da, db, idesc, (i > 0 || it > 0) ? 1u : 0u);
                }
                tc::commit(&empty[s]);
            }
            tc::commit(&acc_full[acc]);  // arrives once every MMA issued above has completed
        }
        tc::commit(done);
    } else if (warp >= 2) {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (rows of the tile), 32 columns at a time, adds
        // the bias and applies ReLU (or writes a split-K partial), and passes them through a 32 x 33
        // transpose in shared memory so that each store instruction writes 32 consecutive columns of a row
        const int quarter = warp % 4;
        float* stage = epi + (warp - 2) * (32 * 33);
        uint32_t j = 0;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++j) {
            const Tile tl = tile_of(t);
            const uint32_t acc = j & 1u;
            ok = mbar_wait_bounded(&acc_full[acc], (j / 2) & 1);
            if (!ok) break;
            tc::fence_after_sync();
            float* cbase = g.c + tl.z * g.split_stride;
            const int64_t mw = tl.m0 + 32 * quarter;
            const int rows = static_cast<int>(min(static_cast<int64_t>(32), g.M - mw));
#pragma unroll 1
            for (int cb = 0; cb < kBN / 32; ++cb) {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tmem + acc * kBN + ((static_cast<uint32_t>(32 * quarter)) << 16) +
                                           static_cast<uint32_t>(32 * cb),
                                       r);
                tc::tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c)  // an empty reduction range contributes zero
                    stage[lane * 33 + c] = tl.nk == 0 ? 0.0f : __uint_as_float(r[c]);
                __syncwarp();
                const int64_t n = tl.n0 + 32 * cb + lane;
                const bool col = n < g.N;
                const float bias = (col && g.bias != nullptr) ? __ldg(g.bias + n) : 0.0f;
                for (int i = 0; i < rows; ++i) {
                    if (col) {
                        float v = stage[i * 33 + lane];
                        if (g.bias != nullptr) v += bias;
                        if (g.relu) v = fmaxf(v, 0.0f);
                        cbase[(mw + i) * g.ldc + n] = v;
                    }
                }
                __syncwarp();  // the stage is rewritten by the next column block
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);  // the accumulator may take tile j + 2
        }
    }
    __syncwarp();
    tc::fence_before_sync();
    ok = mbar_wait_bounded(done, 0) && ok;  // every MMA of this CTA has completed
    ok = __syncthreads_and(ok) != 0;
    if (!ok && threadIdx.x == 0) flag_status(g.status, DLRM_ERR_TIMEOUT);
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 2 * kBN);
    }
}

// ---- operand preparation: fp32 -> bf16 hi / lo ---------------------------------------------------------
__device__ __forceinline__ void split_one(float v, __nv_bfloat16& h, __nv_bfloat16& l)
{
    h = __float2bfloat16_rn(v);
    l = __float2bfloat16_rn(v - __bfloat162float(h));
}

// hi and lo of 8 values as two 16-byte words of bf16 pairs.
__device__ __forceinline__ void split8(const float (&v)[8], uint4& h, uint4& l)
{
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat16 h0, l0, h1, l1;
        split_one(v[2 * i], h0, l0);
        split_one(v[2 * i + 1], h1, l1);
        hw[i] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
        lw[i] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
    }
    h = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    l = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// hi / lo [R x Kp] of src [R x K] (leading dimension ld), times [mask > 0] when a mask (same layout) is
// given; columns K .. Kp - 1 are zero.  A thread splits 8 consecutive columns of a row (Kp is a multiple of
// 8) and stores 16 bytes of hi and 16 of lo; vec: rows start 16-byte aligned, so full groups load as float4.
__global__ void __launch_bounds__(256) split_rows_kernel(const float* __restrict__ src, const float* __restrict__ mask,
                                                         int64_t ld, int64_t R, int64_t K, int64_t Kp, int vec,
                                                         __nv_bfloat16* __restrict__ hi, __nv_bfloat16* __restrict__ lo)
{
    const int64_t groups = Kp / 8;
    const int64_t n = R * groups;
    for (int64_t e = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; e < n; e += int64_t{gridDim.x} * blockDim.x) {
        const int64_t r = e / groups, k0 = (e - r * groups) * 8;
        const float* sr = src + r * ld + k0;
        const float* mr = mask != nullptr ? mask + r * ld + k0 : nullptr;
        float v[8];
        if (vec && k0 + 8 <= K) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(sr)), b = __ldg(reinterpret_cast<const float4*>(sr) + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            if (mr != nullptr) {
                const float4 c = __ldg(reinterpret_cast<const float4*>(mr)), d = __ldg(reinterpret_cast<const float4*>(mr) + 1);
                const float m[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (!(m[i] > 0.0f)) v[i] = 0.0f;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[i] = k0 + i < K ? __ldg(sr + i) : 0.0f;
                if (mr != nullptr && k0 + i < K && !(__ldg(mr + i) > 0.0f)) v[i] = 0.0f;
            }
        }
        uint4 h, l;
        split8(v, h, l);
        reinterpret_cast<uint4*>(hi + r * Kp + k0)[0] = h;
        reinterpret_cast<uint4*>(lo + r * Kp + k0)[0] = l;
    }
}

// The backward's dz = src * [mask > 0] split into hi / lo [R x Kp] (as split_rows_kernel does) and, in the
// same pass, its column sums over row chunks, part[chunk][c] (the bias gradient's partials, added in chunk
// order by the update): per column, row lane ty adds rows r_lo + ty, + 8, ... of the chunk in order, then
// the 8 row lanes are added in order.  A block holds 32 groups of 8 columns x 8 row lanes; enough chunks
// that the batch keeps every SM busy.
constexpr int kColChunks = 256;
__global__ void __launch_bounds__(256) split_rows_colsum_kernel(const float* __restrict__ src,
                                                                const float* __restrict__ mask, int64_t ld, int64_t R,
                                                                int64_t K, int64_t Kp, int vec,
                                                                __nv_bfloat16* __restrict__ hi,
                                                                __nv_bfloat16* __restrict__ lo, float* __restrict__ part)
{
    __shared__ float acc[8][32 * 8 + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t k0 = (static_cast<int64_t>(blockIdx.x) * 32 + tx) * 8;
    const int64_t per = (R + kColChunks - 1) / kColChunks;
    const int64_t r_lo = static_cast<int64_t>(blockIdx.y) * per, r_hi = min(R, r_lo + per);
    float sum[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sum[i] = 0.0f;
    if (k0 < Kp) {
        for (int64_t r = r_lo + ty; r < r_hi; r += 8) {
            const float* sr = src + r * ld + k0;
            const float* mr = mask != nullptr ? mask + r * ld + k0 : nullptr;
            float v[8];
            if (vec && k0 + 8 <= K) {
                const float4 a = __ldg(reinterpret_cast<const float4*>(sr)), b = __ldg(reinterpret_cast<const float4*>(sr) + 1);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
                if (mr != nullptr) {
                    const float4 c = __ldg(reinterpret_cast<const float4*>(mr)), d = __ldg(reinterpret_cast<const float4*>(mr) + 1);
                    const float m[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (!(m[i] > 0.0f)) v[i] = 0.0f;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[i] = k0 + i < K ? __ldg(sr + i) : 0.0f;
                    if (mr != nullptr && k0 + i < K && !(__ldg(mr + i) > 0.0f)) v[i] = 0.0f;
                }
            }
            uint4 h, l;
            split8(v, h, l);
            reinterpret_cast<uint4*>(hi + r * Kp + k0)[0] = h;
            reinterpret_cast<uint4*>(lo + r * Kp + k0)[0] = l;
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[i] += v[i];
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[ty][tx * 8 + i] = sum[i];
    __syncthreads();
    const int64_t c = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    if (c < K) {
        float t = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) t += acc[q][threadIdx.x];
        part[static_cast<int64_t>(blockIdx.y) * K + c] = t;
    }
}

// W -= lr * sum_s partial[s] (splits added in order); b -= lr * sum_chunk db_part[chunk]: a warp per
// element of b, lane l adding chunks l, l + 32, ... in order, then the lanes' sums by a fixed butterfly.
__global__ void __launch_bounds__(256) sgd_update_kernel(float* __restrict__ w, const float* __restrict__ partial,
                                                         int splits, int64_t n, float* __restrict__ b,
                                                         const float* __restrict__ db_part, int64_t nb, float lr)
{
    for (int64_t i = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; i < n; i += int64_t{gridDim.x} * blockDim.x) {
        float s = 0.0f;
        for (int z = 0; z < splits; ++z) s += partial[static_cast<int64_t>(z) * n + i];
        w[i] = fmaf(-lr, s, w[i]);
    }
    if (b != nullptr) {
        const int lane = threadIdx.x % kWarp;
        const int64_t warps = int64_t{gridDim.x} * (blockDim.x / kWarp);
        for (int64_t i = blockIdx.x * int64_t{blockDim.x / kWarp} + threadIdx.x / kWarp; i < nb; i += warps) {
            float s = 0.0f;
            for (int q = lane; q < kColChunks; q += kWarp) s += db_part[static_cast<int64_t>(q) * nb + i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
            if (lane == 0) b[i] = fmaf(-lr, s, b[i]);
        }
    }
}

// ---- head ----------------------------------------------------------------------------------------------
constexpr int kHeadThreads = 256;  // 8 warps, a warp per sample
constexpr int kHeadMaxIn = 1024;

// Per block: its samples' dz h (in_dim values), dz and loss terms, added in sample order.
__global__ void __launch_bounds__(kHeadThreads) head_kernel(const float* __restrict__ h, const float* __restrict__ w,
                                                            const float* __restrict__ b, const float* __restrict__ label,
                                                            int64_t M, int in_dim, int rows_per_block,
                                                            float* __restrict__ prob, float* __restrict__ dh,
                                                            float* __restrict__ part_w, float* __restrict__ part_s)
{
    __shared__ float dz_s[kHeadThreads / kWarp];
    __shared__ float loss_s[kHeadThreads / kWarp];
    __shared__ float acc_w[kHeadThreads / kWarp][kHeadMaxIn];
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * rows_per_block;
    const float bias = __ldg(b);
    for (int k = lane; k < in_dim; k += kWarp) acc_w[warp][k] = 0.0f;
    float dz_sum = 0.0f, loss_sum = 0.0f;
    for (int i = warp; i < rows_per_block; i += kHeadThreads / kWarp) {
        const int64_t m = first + i;
        if (m >= M) break;
        const float* hr = h + m * in_dim;
        float s = 0.0f;
        for (int k = lane; k < in_dim; k += kWarp) s = fmaf(hr[k], __ldg(w + k), s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
        const float z = s + bias;
        const float y = __ldg(label + m);
        const float p = 1.0f / (1.0f + expf(-z));
        const float loss = fmaxf(z, 0.0f) - z * y + log1pf(expf(-fabsf(z)));
        const float dz = (p - y) / static_cast<float>(M);
        if (lane == 0 && prob != nullptr) prob[m] = p;
        float* dr = dh + m * in_dim;
        for (int k = lane; k < in_dim; k += kWarp) {
            dr[k] = dz * __ldg(w + k);
            acc_w[warp][k] = fmaf(dz, hr[k], acc_w[warp][k]);
        }
        dz_sum += dz;
        loss_sum += loss;
    }
    if (lane == 0) {
        dz_s[warp] = dz_sum;
        loss_s[warp] = loss_sum;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < in_dim; k += kHeadThreads) {
        float s = 0.0f;
#pragma unroll
        for (int q = 0; q < kHeadThreads / kWarp; ++q) s += acc_w[q][k];
        part_w[static_cast<int64_t>(blockIdx.x) * in_dim + k] = s;
    }
    if (threadIdx.x == 0) {
        float a = 0.0f, l = 0.0f;
        for (int q = 0; q < kHeadThreads / kWarp; ++q) {
            a += dz_s[q];
            l += loss_s[q];
        }
        part_s[2 * blockIdx.x] = a;
        part_s[2 * blockIdx.x + 1] = l;
    }
}

// Sums the blocks' partials; loss = sum / M; w -= lr dw; b -= lr db.  A warp per element of w (warp K:
// db and the loss): lane l adds blocks l, l + 32, ... in order, then the lanes' sums by a fixed butterfly.
__global__ void __launch_bounds__(256) head_update_kernel(float* __restrict__ w, float* __restrict__ b,
                                                          const float* __restrict__ part_w,
                                                          const float* __restrict__ part_s, int blocks, int in_dim,
                                                          int64_t M, float lr, float* __restrict__ loss)
{
    const int lane = threadIdx.x % kWarp;
    const int k = static_cast<int>(blockIdx.x) * (blockDim.x / kWarp) + static_cast<int>(threadIdx.x / kWarp);
    if (k > in_dim) return;
    float s0 = 0.0f, s1 = 0.0f;
    for (int q = lane; q < blocks; q += kWarp) {
        if (k < in_dim) {
            s0 += part_w[static_cast<int64_t>(q) * in_dim + k];
        } else {
            s0 += part_s[2 * q];
            s1 += part_s[2 * q + 1];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(kFull, s0, o);
        s1 += __shfl_xor_sync(kFull, s1, o);
    }
    if (lane != 0) return;
    if (k < in_dim) {
        w[k] = fmaf(-lr, s0, w[k]);
    } else {
        b[0] = fmaf(-lr, s0, b[0]);
        if (loss != nullptr) loss[0] = s1 / static_cast<float>(M);
    }
}

constexpr int kHeadRowsPerBlock = 64;

inline size_t align256(size_t x) { return (x + 255) & ~size_t{255}; }

int splits_for(int64_t tiles, int64_t K)
{
    // enough CTAs for one per SM (a CTA holds 192 KB of shared memory), each split at least 4 slices of K
    const int sms = sm_count();
    int s = static_cast<int>((static_cast<int64_t>(sms) + tiles - 1) / (tiles > 0 ? tiles : 1));
    const int64_t max_s = (K + 4 * kBK - 1) / (4 * kBK);
    if (s > max_s) s = static_cast<int>(max_s);
    return s < 1 ? 1 : s;
}

int64_t pad8(int64_t x) { return (x + 7) / 8 * 8; }

// cuTensorMapEncodeTiled, resolved once through the runtime (a driver function, the same for every device).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder()
{
    static std::atomic<void*> fn{nullptr};
    void* f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<EncodeFn>(f);
}

// A split operand in global memory: bf16 hi / lo [outer x inner] row-major (inner a multiple of 8).  K-major:
// outer = M (or N) rows of K values; MN-major: outer = K rows of M (or N) values.
struct Operand {
    const __nv_bfloat16 *hi, *lo;
    int64_t inner, outer;
    int mn;
};

// Tiles of 64 inner x (128 rows K-major, 64 rows MN-major), 128-byte swizzle, zero fill out of range.
bool encode_operand(CUtensorMap* map, const __nv_bfloat16* base, const Operand& op)
{
    EncodeFn enc = encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(op.inner), static_cast<cuuint64_t>(op.outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(op.inner) * 2};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(op.mn ? kBK : kBM)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// C[M x N] = A B^T (A: M x K, B: N x K, each K-major or MN-major), K the reduction length; splits > 1: split-K
// partials split_stride elements apart.
dlrm_status launch_gemm(const Operand& A, const Operand& B, const float* bias, float* c, int64_t ldc, int64_t M,
                        int64_t N, int64_t K, int relu, int splits, int64_t split_stride, int32_t* status,
                        cudaStream_t s)
{
    if (M <= 0 || N <= 0) return DLRM_OK;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX || A.inner > INT32_MAX || B.inner > INT32_MAX)
        return DLRM_ERR_UNSUPPORTED;
    GemmArgs g;
    memset(&g, 0, sizeof g);
    if (!encode_operand(&g.a_hi, A.hi, A) || !encode_operand(&g.a_lo, A.lo, A) || !encode_operand(&g.b_hi, B.hi, B) ||
        !encode_operand(&g.b_lo, B.lo, B))
        return DLRM_ERR_CUDA;
    g.a_mn = A.mn;
    g.b_mn = B.mn;
    g.bias = bias;
    g.c = c;
    g.ldc = ldc;
    g.M = M;
    g.N = N;
    g.K = K;
    const int64_t per = (K + splits - 1) / splits;
    g.k_per_split = (per + kBK - 1) / kBK * kBK;
    g.splits = splits;
    g.split_stride = split_stride;
    g.relu = relu;
    g.status = status;
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem) != cudaSuccess)
        return DLRM_ERR_CUDA;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN) * splits;
    const int sms = sm_count();
    if (sms <= 0) return DLRM_ERR_CUDA;
    const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);  // one CTA per SM (shared memory)
    gemm_tc_kernel<<<grid, kGThreads, kGemmSmem, s>>>(g);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

// Carves bf16 hi / lo pairs and fp32 arrays out of a workspace, 256-byte aligned.
struct Carver {
    char* p;
    size_t used = 0;
    template <typename T>
    T* take(size_t count)
    {
        T* at = p ? reinterpret_cast<T*>(p + used) : nullptr;
        used = align256(used + sizeof(T) * count);
        return at;
    }
};

void split_rows(const float* src, const float* mask, int64_t ld, int64_t R, int64_t K, int64_t Kp, __nv_bfloat16* hi,
                __nv_bfloat16* lo, cudaStream_t s)
{
    const int64_t n = R * (Kp / 8);
    const int64_t blocks = (n + 255) / 256;
    const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const int vec = ld % 4 == 0 && a16(src) && (mask == nullptr || a16(mask));
    split_rows_kernel<<<static_cast<unsigned>(blocks < 148 * 16 ? blocks : 148 * 16), 256, 0, s>>>(src, mask, ld, R, K,
                                                                                                   Kp, vec, hi, lo);
}

// Workspace of the forward: x and W split.
struct FwdWs {
    __nv_bfloat16 *xh, *xl, *wh, *wl;
};
FwdWs carve_fwd(void* base, int64_t M, int32_t K, int32_t N, size_t* bytes)
{
    Carver c{static_cast<char*>(base)};
    const int64_t kp = pad8(K);
    FwdWs w;
    w.xh = c.take<__nv_bfloat16>(M * kp);
    w.xl = c.take<__nv_bfloat16>(M * kp);
    w.wh = c.take<__nv_bfloat16>(static_cast<int64_t>(N) * kp);
    w.wl = c.take<__nv_bfloat16>(static_cast<int64_t>(N) * kp);
    if (bytes) *bytes = c.used;
    return w;
}

// Workspace of the backward: dz, W and x split once (row by row); dx and dW read them K-major or MN-major as
// each product needs; the dW partials, the db partials.
struct BwdWs {
    __nv_bfloat16 *dzh, *dzl, *wh, *wl, *xh, *xl;
    float *part, *db_part;
    int splits;
};
BwdWs carve_bwd(void* base, int64_t M, int32_t K, int32_t N, size_t* bytes)
{
    Carver c{static_cast<char*>(base)};
    const int64_t np = pad8(N), kp = pad8(K);
    BwdWs w;
    const int64_t tiles = ((N + kBM - 1) / kBM) * ((K + kBN - 1) / kBN);
    w.splits = splits_for(tiles, M);
    w.dzh = c.take<__nv_bfloat16>(M * np);
    w.dzl = c.take<__nv_bfloat16>(M * np);
    w.wh = c.take<__nv_bfloat16>(static_cast<int64_t>(N) * kp);
    w.wl = c.take<__nv_bfloat16>(static_cast<int64_t>(N) * kp);
    w.xh = c.take<__nv_bfloat16>(M * kp);
    w.xl = c.take<__nv_bfloat16>(M * kp);
    w.part = c.take<float>(static_cast<size_t>(w.splits) * N * K);
    w.db_part = c.take<float>(static_cast<size_t>(kColChunks) * N);
    if (bytes) *bytes = c.used;
    return w;
}

}  // namespace

size_t fc_fwd_workspace_bytes(int64_t M, int32_t K, int32_t N)
{
    size_t b = 0;
    carve_fwd(nullptr, M, K, N, &b);
    return b;
}

size_t fc_bwd_workspace_bytes(int64_t M, int32_t K, int32_t N)
{
    size_t b = 0;
    carve_bwd(nullptr, M, K, N, &b);
    return b;
}

dlrm_status launch_fc_fwd(const float* x, const float* w, const float* b, int64_t M, int32_t K, int32_t N, int relu,
                          float* y, void* workspace, int32_t* status, cudaStream_t s)
{
    const FwdWs ws = carve_fwd(workspace, M, K, N, nullptr);
    const int64_t kp = pad8(K);
    split_rows(x, nullptr, K, M, K, kp, ws.xh, ws.xl, s);
    split_rows(w, nullptr, K, N, K, kp, ws.wh, ws.wl, s);
    // y = x W^T: A = x [M x K], B = W [N x K], both K-major
    const Operand A{ws.xh, ws.xl, kp, M, 0}, B{ws.wh, ws.wl, kp, N, 0};
    return launch_gemm(A, B, b, y, N, M, N, K, relu, 1, 0, status, s);
}

dlrm_status launch_fc_bwd_sgd(const float* x, float* w, float* b, const float* y, const float* dy, int64_t M, int32_t K,
                              int32_t N, int relu, float lr, float* dx, void* workspace, int32_t* status,
                              cudaStream_t s)
{
    const BwdWs ws = carve_bwd(workspace, M, K, N, nullptr);
    const int64_t np = pad8(N), kp = pad8(K);
    const float* mask = relu ? y : nullptr;
    if (b != nullptr) {  // dz = dy [y > 0], [M x N], and the partials of db = sum over the batch of dz
        const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
        const int vec = N % 4 == 0 && a16(dy) && (mask == nullptr || a16(mask));
        const dim3 grid(static_cast<unsigned>((np / 8 + 31) / 32), kColChunks);
        split_rows_colsum_kernel<<<grid, 256, 0, s>>>(dy, mask, N, M, N, np, vec, ws.dzh, ws.dzl, ws.db_part);
    } else {
        split_rows(dy, mask, N, M, N, np, ws.dzh, ws.dzl, s);
    }
    split_rows(x, nullptr, K, M, K, kp, ws.xh, ws.xl, s);  // x [M x K]
    // dx = dz W: A = dz [M x N] K-major; B[k][n] = W[n][k]: W [N x K] read MN-major
    if (dx != nullptr) {
        split_rows(w, nullptr, K, N, K, kp, ws.wh, ws.wl, s);
        const Operand A{ws.dzh, ws.dzl, np, M, 0}, B{ws.wh, ws.wl, kp, N, 1};
        dlrm_status st = launch_gemm(A, B, nullptr, dx, K, M, K, N, 0, 1, 0, status, s);
        if (st != DLRM_OK) return st;
    }
    // dW = dz^T x over the batch, in split partials: A[n][m] = dz[m][n], B[k][m] = x[m][k], both read MN-major
    const Operand A{ws.dzh, ws.dzl, np, M, 1}, B{ws.xh, ws.xl, kp, M, 1};
    dlrm_status st = launch_gemm(A, B, nullptr, ws.part, K, N, K, M, 0, ws.splits, static_cast<int64_t>(N) * K, status, s);
    if (st != DLRM_OK) return st;
    const int64_t n = static_cast<int64_t>(N) * K;
    const int64_t blocks = (n + 255) / 256;
    sgd_update_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(
        w, ws.part, ws.splits, n, b, ws.db_part, b != nullptr ? N : 0, lr);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

size_t head_workspace_bytes(int64_t M, int32_t K)
{
    const int64_t blocks = (M + kHeadRowsPerBlock - 1) / kHeadRowsPerBlock;
    return align256(sizeof(float) * static_cast<size_t>(blocks) * K) + align256(sizeof(float) * 2 * blocks);
}

dlrm_status launch_head(const float* h, float* w, float* b, const float* label, int64_t M, int32_t K, float lr,
                        float* prob, float* loss, float* dh, void* workspace, cudaStream_t s)
{
    if (K > kHeadMaxIn) return DLRM_ERR_UNSUPPORTED;
    const int64_t blocks = (M + kHeadRowsPerBlock - 1) / kHeadRowsPerBlock;
    if (blocks > 0x7fffffff) return DLRM_ERR_UNSUPPORTED;
    float* part_w = static_cast<float*>(workspace);
    float* part_s = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             align256(sizeof(float) * static_cast<size_t>(blocks) * K));
    head_kernel<<<static_cast<unsigned>(blocks), kHeadThreads, 0, s>>>(h, w, b, label, M, K, kHeadRowsPerBlock, prob,
                                                                       dh, part_w, part_s);
    head_update_kernel<<<static_cast<unsigned>((K + 1 + 7) / 8), 256, 0, s>>>(w, b, part_w, part_s,
                                                                               static_cast<int>(blocks), K, M, lr, loss);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

}  // namespace dlrm
