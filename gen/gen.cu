// gen.cu -- counter-based table-content generator, host loop and device fill.
//
// Input generation only: this file holds none of the DLRM arithmetic.  It is
// shared by the tests and the benchmark; the product library does not link it.
// The definition (SplitMix64 of Steele, Lea & Flood, OOPSLA 2014, used as a
// counter-based hash) is written out in gen/__init__.py, whose numpy version
// is the reference the two fills here are checked against bit for bit.
#include <cuda_runtime.h>
#include <omp.h>
#include <stdint.h>
#include <string.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// fp32(0.1) * 2^-24, exact.
__host__ __device__ inline float value_scale() { return 0.100000001490116119384765625f / 16777216.0f; }

__host__ __device__ inline float elem_value(uint64_t stream, uint64_t counter)
{
    uint64_t h = mix64(stream + (counter + 1) * kGamma);
    int32_t k = (int32_t)(h >> 40) - (1 << 23);
#ifdef __CUDA_ARCH__
    return __fmul_rn((float)k, value_scale());
#else
    return (float)k * value_scale();  // one fp32 multiply, round to nearest even
#endif
}

__host__ __device__ inline uint16_t to_bf16_rne(float v)
{
    uint32_t bits;
#ifdef __CUDA_ARCH__
    bits = __float_as_uint(v);
#else
    memcpy(&bits, &v, 4);
#endif
    return (uint16_t)((bits + 0x7FFFu + ((bits >> 16) & 1u)) >> 16);
}

__global__ void fill_kernel(void* dst, int bf16, uint64_t stream, int64_t row0, int64_t nrows, int D)
{
    const int64_t n = nrows * (int64_t)D;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t counter = (uint64_t)(row0 * (int64_t)D + i);
        const float v = elem_value(stream, counter);
        if (bf16)
            static_cast<uint16_t*>(dst)[row0 * (int64_t)D + i] = to_bf16_rne(v);
        else
            static_cast<float*>(dst)[row0 * (int64_t)D + i] = v;
    }
}

}  // namespace

extern "C" {

// Rows rows[0..n) of one table (stream key `stream`) into out[n][D]
// (float32, or bf16 bit patterns when bf16 != 0).  threads <= 0: all cores.
void gen_rows_host(void* out, int bf16, uint64_t stream, const int64_t* rows, int64_t n, int D, int threads)
{
    const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t i = 0; i < n; ++i) {
        const uint64_t base = (uint64_t)rows[i] * (uint64_t)D;
        for (int d = 0; d < D; ++d) {
            const float v = elem_value(stream, base + (uint64_t)d);
            if (bf16)
                static_cast<uint16_t*>(out)[i * D + d] = to_bf16_rne(v);
            else
                static_cast<float*>(out)[i * D + d] = v;
        }
    }
}

// Fill rows [row0, row0+nrows) of a row-major table at device pointer dst.
// Returns 0 or the CUDA error code of the launch.
int gen_fill_device(void* dst, int bf16, uint64_t stream, int64_t row0, int64_t nrows, int D, cudaStream_t s)
{
    if (nrows <= 0) return 0;
    const int64_t n = nrows * (int64_t)D;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 148 * 64) blocks = 148 * 64;
    fill_kernel<<<(unsigned)blocks, 256, 0, s>>>(dst, bf16, stream, row0, nrows, D);
    return (int)cudaGetLastError();
}

}  // extern "C"
