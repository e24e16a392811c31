// mlp.cu -- the dense layers around the sparse path: the bottom MLP, the top
// MLP and the sigmoid output with its binary cross-entropy loss, forward and
// backward with plain SGD on their weights ("DLRM", robocikowo.com, "Forward
// pass" steps (1) and (4), the bottom-MLP and top-MLP paragraphs: FC layers
// with ReLU, a sigmoid output; the hardware paragraph: the MLPs are ordinary
// GEMMs on the tensor cores).
//
// GEMM.  C[M x N] = A[M x K] * B[N x K]^T with both operands K-major in global
// memory (a row of A or B holds its K values contiguously), on the tcgen05
// tensor cores: a CTA of 256 threads owns a 128 x 128 tile of C, walks K in
// slices of 64, double-buffered in shared memory.  The threads load a slice of
// fp32 A and B rows (16-byte loads where the rows allow), split each value v
// into bf16 hi = bf16(v) and lo = bf16(v - hi) and store both into K-major
// 128-byte-swizzled operand buffers; one thread issues hi*hi^T + hi*lo^T +
// lo*hi^T (3 x 4 MMAs of 128 x 128 x 16) into a 128-column fp32 accumulator in
// TMEM and commits them to the slice's mbarrier, while the threads load the
// next slice.  The dropped lo*lo term and the rounding of lo stay below 2^-16
// relative to sum |a_k b_k|.  Epilogue: warp w reads TMEM lanes
// 32 (w % 4) .. + 31 (rows of C), columns 64 (w / 4) .. + 63, adds the bias and
// applies ReLU, or writes a split-K partial.
//
// Backward of y = act(x W^T + b) from dy: dz = dy * [y > 0] (ReLU) or dy;
// dx = dz W; dW = dz^T x; db = sum over the batch of dz.  dx is a GEMM with A =
// dz (the mask applied while A is loaded) and B = W^T (an explicit transpose of
// the small W); dW is a GEMM over the batch with A = dz^T and B = x^T (tiled
// transposes through shared memory, the mask applied in the transpose), split
// over the batch into partial sums that the update kernel adds in a fixed order
// (bitwise reproducible) before W -= lr dW, b -= lr db.
//
// Head.  The last top layer maps to one logit: a warp per sample computes
// z = h . w + b, p = sigmoid(z), the sample's BCE term max(z, 0) - z y +
// log(1 + exp(-|z|)) and dz = (p - y) / M, writes dh = dz w, and the block adds
// its samples' dz h, dz and loss terms in a fixed order; a reduce kernel sums the
// blocks' partials in order, writes the mean loss and applies SGD to w and b.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dlrm {
namespace {

constexpr int kGThreads = 256;
constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kSlice = kBM * kBK * 2;  // one bf16 operand slice, 16 KB (kBM == kBN)
constexpr int kStage = 4 * kSlice;     // A hi, A lo, B hi, B lo
constexpr int kGemmSmem = 2 * kStage + 1024 + 64;
constexpr uint32_t kFull = 0xffffffffu;

struct GemmArgs {
    const float* a;
    const float* amask;  // optional: A multiplied by [amask > 0] (same layout, leading dimension lda)
    const float* b;
    const float* bias;   // optional, N values
    float* c;
    int64_t lda, ldb, ldc;
    int64_t M, N, K;
    int64_t k_per_split;   // reduction range of split z: [z * k_per_split, min(K, (z + 1) * k_per_split))
    int64_t split_stride;  // elements between the C partials of consecutive splits
    int relu;
    int vec_a, vec_b;      // 16-byte loads allowed
    int32_t* status;
};

// Byte offset of (row, byte b of its 128-byte K extent) in a K-major 128-byte-swizzle operand slice.
__device__ __forceinline__ uint32_t sw128(int row, int b)
{
    return row * 128 + ((((b >> 4) ^ (row & 7)) << 4) | (b & 15));
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 h)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(h.x)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h.y)) << 16);
}

__device__ __forceinline__ void split_store(unsigned char* hi, unsigned char* lo, int row, int kc, float4 v)
{
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
    const uint32_t off = sw128(row, kc * 8);
    *reinterpret_cast<uint2*>(hi + off) = make_uint2(bf16x2_bits(h01), bf16x2_bits(h23));
    *reinterpret_cast<uint2*>(lo + off) = make_uint2(bf16x2_bits(l01), bf16x2_bits(l23));
}

// Rows r0 .. r0 + 127 (below R) and K values k0 .. k0 + 63 (below kend) of a K-major fp32 matrix into the
// hi / lo slices; 8 float4 per thread, every load issued before the splits.
__device__ __forceinline__ void load_slice(const float* src, const float* mask, int64_t ld, int vec, int64_t r0,
                                           int64_t R, int64_t k0, int64_t kend, unsigned char* hi, unsigned char* lo)
{
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = threadIdx.x + i * kGThreads;
        const int row = idx >> 4, kc = idx & 15;
        const int64_t r = r0 + row, k = k0 + kc * 4;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < R) {
            const float* p = src + r * ld + k;
            if (vec && k + 3 < kend) {
                v[i] = __ldg(reinterpret_cast<const float4*>(p));
                if (mask != nullptr) {
                    const float4 m = __ldg(reinterpret_cast<const float4*>(mask + r * ld + k));
                    v[i] = make_float4(m.x > 0.f ? v[i].x : 0.f, m.y > 0.f ? v[i].y : 0.f, m.z > 0.f ? v[i].z : 0.f,
                                       m.w > 0.f ? v[i].w : 0.f);
                }
            } else {
                float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (k + j < kend) {
                        e[j] = __ldg(p + j);
                        if (mask != nullptr && !(__ldg(mask + r * ld + k + j) > 0.f)) e[j] = 0.f;
                    }
                v[i] = make_float4(e[0], e[1], e[2], e[3]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = threadIdx.x + i * kGThreads;
        split_store(hi, lo, idx >> 4, idx & 15, v[i]);
    }
}

__global__ void __launch_bounds__(kGThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmArgs g)
{
    extern __shared__ unsigned char gsm_raw[];
    unsigned char* sm = gsm_raw + ((1024u - (smem_addr(gsm_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 2 * kStage);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + 2 * kStage + 16);
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kBM, n0 = static_cast<int64_t>(blockIdx.y) * kBN;
    const int64_t kb = static_cast<int64_t>(blockIdx.z) * g.k_per_split;
    const int64_t ke = min(g.K, kb + g.k_per_split);
    const int nk = ke > kb ? static_cast<int>((ke - kb + kBK - 1) / kBK) : 0;

    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kBN);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    auto stage_ptr = [&](int s, int which) { return sm + s * kStage + which * kSlice; };
    bool ok = true;
    if (nk > 0) {
        load_slice(g.a, g.amask, g.lda, g.vec_a, m0, g.M, kb, ke, stage_ptr(0, 0), stage_ptr(0, 1));
        load_slice(g.b, nullptr, g.ldb, g.vec_b, n0, g.N, kb, ke, stage_ptr(0, 2), stage_ptr(0, 3));
    }
    for (int i = 0; i < nk; ++i) {
        const int s = i & 1;
        tc::fence_smem_for_mma();
        __syncthreads();
        if (threadIdx.x == 0) {
            tc::fence_after_sync();
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
            const uint32_t a_hi = smem_addr(stage_ptr(s, 0)), a_lo = smem_addr(stage_ptr(s, 1));
            const uint32_t b_hi = smem_addr(stage_ptr(s, 2)), b_lo = smem_addr(stage_ptr(s, 3));
#pragma unroll
            for (int it = 0; it < 12; ++it) {  // hi*hi, hi*lo, lo*hi over 4 steps of K = 16
                const int pass = it / 4, ks = it % 4;
                const uint32_t A = (pass == 2 ? a_lo : a_hi) + ks * 32;
                const uint32_t B = (pass == 1 ? b_lo : b_hi) + ks * 32;
                tc::mma_bf16(tmem, tc::desc_kmajor_sw128(A), tc::desc_kmajor_sw128(B), idesc, (i > 0 || it > 0) ? 1u : 0u);
            }
            tc::commit(&bar[s]);
        }
        if (i + 1 < nk) {
            const int s2 = (i + 1) & 1;
            if (i >= 1) ok &= mbar_wait_bounded(&bar[s2], ((i - 1) >> 1) & 1);  // slice i - 1 read by the MMAs
            const int64_t k0 = kb + static_cast<int64_t>(i + 1) * kBK;
            load_slice(g.a, g.amask, g.lda, g.vec_a, m0, g.M, k0, ke, stage_ptr(s2, 0), stage_ptr(s2, 1));
            load_slice(g.b, nullptr, g.ldb, g.vec_b, n0, g.N, k0, ke, stage_ptr(s2, 2), stage_ptr(s2, 3));
        }
    }
    if (nk > 0) ok &= mbar_wait_bounded(&bar[(nk - 1) & 1], ((nk - 1) >> 1) & 1);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
        if (threadIdx.x == 0 && nk > 0) {
            flag_status(g.status, DLRM_ERR_TIMEOUT);
            (void)mbar_wait_bounded(&bar[(nk - 1) & 1], ((nk - 1) >> 1) & 1);  // the MMAs still in flight end first
        }
        __syncthreads();
    }
    tc::fence_after_sync();

    // epilogue: rows 32 (warp % 4) + lane, columns 64 (warp / 4) .. + 63
    if (ok) {
        const int q = warp & 3, half = warp >> 2;
        const int64_t m = m0 + 32 * q + lane;
        float* crow = g.c + static_cast<int64_t>(blockIdx.z) * g.split_stride + m * g.ldc;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            const int col0 = half * 64 + cb * 32;
            uint32_t r[32];
            tc::tmem_ld_32x32b_x32(tmem + ((static_cast<uint32_t>(32 * q)) << 16) + static_cast<uint32_t>(col0), r);
            tc::tmem_ld_wait();
            if (nk == 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = 0u;  // an empty reduction range contributes zero
            }
            if (m < g.M) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int64_t n = n0 + col0 + j;
                    if (n < g.N) {
                        float v = __uint_as_float(r[j]);
                        if (g.bias != nullptr) v += __ldg(g.bias + n);
                        if (g.relu) v = fmaxf(v, 0.0f);
                        crow[n] = v;
                    }
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kBN);
    }
}

// out[c][r] = in[r][c] (times [mask[r][c] > 0] when a mask is given); in is R x C, out is C x R.
__global__ void __launch_bounds__(256) transpose_kernel(const float* __restrict__ in, const float* __restrict__ mask,
                                                        float* __restrict__ out, int64_t R, int64_t C)
{
    __shared__ float tile[32][33];
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 32, r0 = static_cast<int64_t>(blockIdx.y) * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
    for (int j = ty; j < 32; j += 8) {
        const int64_t r = r0 + j, c = c0 + tx;
        float v = 0.0f;
        if (r < R && c < C) {
            v = in[r * C + c];
            if (mask != nullptr && !(mask[r * C + c] > 0.0f)) v = 0.0f;
        }
        tile[j][tx] = v;
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int64_t c = c0 + j, r = r0 + tx;
        if (c < C && r < R) out[c * R + r] = tile[tx][j];
    }
}

// Row sums of X (rows x cols, cols contiguous), one block per row, a fixed reduction tree.
__global__ void __launch_bounds__(256) row_sum_kernel(const float* __restrict__ x, int64_t cols, float* __restrict__ out)
{
    __shared__ float part[256];
    const float* row = x + static_cast<int64_t>(blockIdx.x) * cols;
    float s = 0.0f;
    for (int64_t c = threadIdx.x; c < cols; c += 256) s += row[c];
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[blockIdx.x] = part[0];
}

// W -= lr * sum_s partial[s] (splits added in order), b -= lr * db.
__global__ void __launch_bounds__(256) sgd_update_kernel(float* __restrict__ w, const float* __restrict__ partial,
                                                         int splits, int64_t n, float* __restrict__ b,
                                                         const float* __restrict__ db, int64_t nb, float lr)
{
    for (int64_t i = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; i < n; i += int64_t{gridDim.x} * blockDim.x) {
        float s = 0.0f;
        for (int z = 0; z < splits; ++z) s += partial[static_cast<int64_t>(z) * n + i];
        w[i] = fmaf(-lr, s, w[i]);
    }
    if (b != nullptr)
        for (int64_t i = blockIdx.x * int64_t{blockDim.x} + threadIdx.x; i < nb; i += int64_t{gridDim.x} * blockDim.x)
            b[i] = fmaf(-lr, db[i], b[i]);
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

// Sums the blocks' partials in block order; loss = sum / M; w -= lr dw; b -= lr db.
__global__ void __launch_bounds__(256) head_update_kernel(float* __restrict__ w, float* __restrict__ b,
                                                          const float* __restrict__ part_w,
                                                          const float* __restrict__ part_s, int blocks, int in_dim,
                                                          int64_t M, float lr, float* __restrict__ loss)
{
    for (int k = threadIdx.x; k < in_dim; k += blockDim.x) {
        float s = 0.0f;
        for (int q = 0; q < blocks; ++q) s += part_w[static_cast<int64_t>(q) * in_dim + k];
        w[k] = fmaf(-lr, s, w[k]);
    }
    if (threadIdx.x == 0) {
        float db = 0.0f, l = 0.0f;
        for (int q = 0; q < blocks; ++q) {
            db += part_s[2 * q];
            l += part_s[2 * q + 1];
        }
        b[0] = fmaf(-lr, db, b[0]);
        if (loss != nullptr) loss[0] = l / static_cast<float>(M);
    }
}

constexpr int kHeadRowsPerBlock = 64;

inline size_t align256(size_t x) { return (x + 255) & ~size_t{255}; }

int splits_for(int64_t tiles, int64_t K)
{
    // enough CTAs for two per SM, each split at least 4 slices of K
    const int sms = sm_count();
    int s = static_cast<int>((2 * static_cast<int64_t>(sms) + tiles - 1) / (tiles > 0 ? tiles : 1));
    const int64_t max_s = (K + 4 * kBK - 1) / (4 * kBK);
    if (s > max_s) s = static_cast<int>(max_s);
    return s < 1 ? 1 : s;
}

}  // namespace

dlrm_status launch_gemm(const float* a, const float* amask, int64_t lda, const float* b, int64_t ldb,
                        const float* bias, float* c, int64_t ldc, int64_t M, int64_t N, int64_t K, int relu,
                        int splits, int64_t split_stride, int32_t* status, cudaStream_t s)
{
    if (M <= 0 || N <= 0) return DLRM_OK;
    GemmArgs g;
    g.a = a;
    g.amask = amask;
    g.b = b;
    g.bias = bias;
    g.c = c;
    g.lda = lda;
    g.ldb = ldb;
    g.ldc = ldc;
    g.M = M;
    g.N = N;
    g.K = K;
    const int64_t per = (K + splits - 1) / splits;
    g.k_per_split = (per + kBK - 1) / kBK * kBK;
    g.split_stride = split_stride;
    g.relu = relu;
    g.vec_a = (lda % 4 == 0) && ((reinterpret_cast<uintptr_t>(a) & 15u) == 0) &&
              (amask == nullptr || (reinterpret_cast<uintptr_t>(amask) & 15u) == 0);
    g.vec_b = (ldb % 4 == 0) && ((reinterpret_cast<uintptr_t>(b) & 15u) == 0);
    g.status = status;
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem) != cudaSuccess)
        return DLRM_ERR_CUDA;
    const dim3 grid(static_cast<unsigned>((M + kBM - 1) / kBM), static_cast<unsigned>((N + kBN - 1) / kBN),
                    static_cast<unsigned>(splits));
    gemm_tc_kernel<<<grid, kGThreads, kGemmSmem, s>>>(g);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

size_t fc_bwd_workspace_bytes(int64_t M, int32_t K, int32_t N)
{
    const int64_t tiles = ((N + kBN - 1) / kBN) * ((K + kBN - 1) / kBN);
    const int splits = splits_for(tiles, M);
    return align256(sizeof(float) * static_cast<size_t>(K) * N)            // W^T
           + align256(sizeof(float) * static_cast<size_t>(N) * M)          // dz^T
           + align256(sizeof(float) * static_cast<size_t>(K) * M)          // x^T
           + align256(sizeof(float) * static_cast<size_t>(splits) * N * K) // dW partials
           + align256(sizeof(float) * static_cast<size_t>(N));             // db
}

dlrm_status launch_fc_fwd(const float* x, const float* w, const float* b, int64_t M, int32_t K, int32_t N, int relu,
                          float* y, int32_t* status, cudaStream_t s)
{
    return launch_gemm(x, nullptr, K, w, K, b, y, N, M, N, K, relu, 1, 0, status, s);
}

dlrm_status launch_fc_bwd_sgd(const float* x, float* w, float* b, const float* y, const float* dy, int64_t M, int32_t K,
                              int32_t N, int relu, float lr, float* dx, void* workspace, int32_t* status,
                              cudaStream_t s)
{
    const int64_t tiles = ((N + kBN - 1) / kBN) * ((K + kBN - 1) / kBN);
    const int splits = splits_for(tiles, M);
    char* p = static_cast<char*>(workspace);
    float* wt = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * static_cast<size_t>(K) * N);
    float* dzt = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * static_cast<size_t>(N) * M);
    float* xt = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * static_cast<size_t>(K) * M);
    float* part = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * static_cast<size_t>(splits) * N * K);
    float* db = reinterpret_cast<float*>(p);
    const float* mask = relu ? y : nullptr;

    auto transpose = [&](const float* in, const float* msk, float* out, int64_t R, int64_t C) {
        const dim3 grid(static_cast<unsigned>((C + 31) / 32), static_cast<unsigned>((R + 31) / 32));
        transpose_kernel<<<grid, 256, 0, s>>>(in, msk, out, R, C);
    };
    // dx = dz W = dz (W^T)^T, with the ReLU mask applied to dz while it is loaded
    if (dx != nullptr) {
        transpose(w, nullptr, wt, N, K);
        dlrm_status st = launch_gemm(dy, mask, N, wt, N, nullptr, dx, K, M, K, N, 0, 1, 0, status, s);
        if (st != DLRM_OK) return st;
    }
    // dW = dz^T x over the batch, in split partials; db = row sums of dz^T
    transpose(dy, mask, dzt, M, N);
    transpose(x, nullptr, xt, M, K);
    dlrm_status st = launch_gemm(dzt, nullptr, M, xt, M, nullptr, part, K, N, K, M, 0, splits,
                                 static_cast<int64_t>(N) * K, status, s);
    if (st != DLRM_OK) return st;
    row_sum_kernel<<<static_cast<unsigned>(N), 256, 0, s>>>(dzt, M, db);
    const int64_t n = static_cast<int64_t>(N) * K;
    const int64_t blocks = (n + 255) / 256;
    sgd_update_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(w, part, splits, n, b, db,
                                                                                          b != nullptr ? N : 0, lr);
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
    head_update_kernel<<<1, 256, 0, s>>>(w, b, part_w, part_s, static_cast<int>(blocks), K, M, lr, loss);
    return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA;
}

}  // namespace dlrm
