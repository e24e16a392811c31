/*
 * dlrm_sparse.h -- C ABI of the DLRM sparse path on one NVIDIA B300 (sm_103a).
 *
 * The path (web pages cited by title and section):
 *   - embedding tables E_t : V_t x D, one per sparse feature ("DLRM",
 *     robocikowo.com, embedding-table paragraph); one lookup per feature
 *     ("DLRM explained", "How does DLRM actually work?"), or several IDs per
 *     feature ("The embedding table is the model"), pooled into one vector;
 *   - the feature interaction: all N = 1 + T vectors (bottom-MLP output x
 *     first, then the T pooled embeddings) as rows of a matrix, pairwise dot
 *     products forming an N x N matrix, of which the strict upper triangle of
 *     N(N-1)/2 values is kept ("DLRM", robocikowo.com, "Forward pass" step (3)
 *     and the interaction-layer paragraph) and concatenated with x ("Forward
 *     pass" step (4); "Deep Learning Recommendation Model (DLRM)",
 *     notes.helloworld.co.in, "The architecture");
 *   - training with Adagrad ("DLRM", robocikowo.com, "Forward pass", last
 *     sentence), here its row-wise form on the embedding rows.
 *
 * Layouts (all row-major, fp32 unless stated):
 *   table t      V_t x D elements (fp32 or bf16), row stride D
 *   bags         CSR, table-major: bag (t,b) = indices[offsets[t*B+b] ..
 *                offsets[t*B+b+1]); indices are rows local to table t;
 *                offsets has T*B+1 entries, offsets[0] = 0, offsets[T*B] = nnz
 *   dense x      B x D
 *   pooled P     B x T x D
 *   out          B x (D + N(N-1)/2): x copied, then z(i,j) = <V_i, V_j> for
 *                0 <= i < j < N in row-major order, i.e. position
 *                i*N - i*(i+1)/2 + (j-i-1) after the first D values;
 *                V_0 = x, V_{1+t} = P[b][t]
 *
 * Conventions shared by every entry point:
 *   - pointers marked "device" must be device memory of the current device;
 *     the caller owns all memory; the library allocates nothing;
 *   - device pointers to tables, dense, pooled, workspace and accumulators
 *     must be 16-byte aligned (cudaMalloc gives 256);
 *   - every call is asynchronous and ordered on `stream`; the return value
 *     reports only what the host can check before launching;
 *   - data errors found on the device (an index outside [0, V_t), a bag range
 *     that is negative, reversed or past nnz, offsets[0] != 0 or
 *     offsets[T*B] != nnz, a device wait that ran out of time) are OR-ed into
 *     *status_dev when status_dev is not NULL; the caller zeroes it before
 *     the call and reads it after synchronising.  An out-of-range lookup
 *     contributes zero (it still counts in a mean's bag length); a bad bag
 *     range is treated as an empty bag.  Kernels never trap;
 *   - outputs must not alias inputs;
 *   - nothing falls back to the CPU.
 */
#ifndef DLRM_SPARSE_H
#define DLRM_SPARSE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status bits: a return value or *status_dev is an OR of these. */
typedef int32_t dlrm_status;
enum {
    DLRM_OK = 0,
    DLRM_ERR_INVALID_ARG = 1,  /* host-checked: null pointer, size out of range, misalignment */
    DLRM_ERR_INDEX_OOB = 2,    /* device: index outside [0, V_t) */
    DLRM_ERR_BAD_OFFSETS = 4,  /* device: malformed CSR offsets */
    DLRM_ERR_TIMEOUT = 8,      /* device: a bounded wait gave up (work of that sample skipped) */
    DLRM_ERR_CUDA = 16,        /* a CUDA launch or copy returned an error */
    DLRM_ERR_UNSUPPORTED = 32  /* valid request the library does not implement */
};

typedef enum { DLRM_POOL_SUM = 0, DLRM_POOL_MEAN = 1 } dlrm_pool_mode;
typedef enum { DLRM_F32 = 0, DLRM_BF16 = 1 } dlrm_dtype;
typedef enum { DLRM_I32 = 0, DLRM_I64 = 1 } dlrm_index_type;

/* Limits of the library. */
#define DLRM_MAX_TABLES 128

/* The embedding tables.  num_tables = T in [1, DLRM_MAX_TABLES]; dim = D in
 * {16, 32, 64, 128, 256}.  data and num_rows are HOST arrays of T entries:
 * data[t] is the device pointer of table t (V_t x D, row stride D, elements
 * of type dtype), num_rows[t] = V_t >= 1. */
typedef struct {
    int32_t num_tables;
    int32_t dim;
    int32_t dtype;              /* dlrm_dtype */
    void *const *data;
    const int64_t *num_rows;
} dlrm_tables;

/* One batch of bags.  batch = B >= 1, nnz >= 0.  indices (device, nnz
 * entries) and offsets (device, T*B+1 entries) share index_type. */
typedef struct {
    int64_t batch;
    int64_t nnz;
    int32_t index_type;         /* dlrm_index_type */
    const void *indices;
    const void *offsets;
} dlrm_bags;

/* Embedding lookup with pooling ("DLRM", robocikowo.com, "Forward pass"
 * step (2); several IDs per feature: "The embedding table is the model").
 *   pooled[b][t][:] = sum (or mean) of E_t[indices[p]][:] over the lookups p
 *                     of bag (t,b), accumulated in fp32; an empty bag gives 0.
 * pooled: device, B x T x D fp32.  status_dev: device int32 or NULL. */
dlrm_status dlrm_embbag_fwd(const dlrm_tables *tables, const dlrm_bags *bags,
                            dlrm_pool_mode mode, float *pooled,
                            int32_t *status_dev, cudaStream_t stream);

/* Feature interaction on given vectors ("DLRM", robocikowo.com, "Forward
 * pass" steps (3)-(4)): out[b] = [x_b, z_b(i,j) for i < j], z in fp32.
 * dense: device B x D; pooled: device B x T x D; out: device B x (D+N(N-1)/2).
 * batch = B >= 1, num_tables = T in [1, DLRM_MAX_TABLES], dim = D as above. */
dlrm_status dlrm_interact_fwd(const float *dense, const float *pooled,
                              int64_t batch, int32_t num_tables, int32_t dim,
                              float *out, cudaStream_t stream);

/* The fused sparse forward: lookup + pooling + interaction + concatenation
 * in one pass; the pooled vectors stay on chip.  Same result as
 * dlrm_embbag_fwd followed by dlrm_interact_fwd.
 * dense: device B x D; out: device B x (D+N(N-1)/2); pooled_save: device
 * B x T x D or NULL (written when given, for the training step). */
dlrm_status dlrm_sparse_fwd(const dlrm_tables *tables, const dlrm_bags *bags,
                            dlrm_pool_mode mode, const float *dense,
                            float *out, float *pooled_save,
                            int32_t *status_dev, cudaStream_t stream);

/* The fused sparse forward fed from HOST memory: copies indices, offsets and
 * dense from host to the caller's device staging buffers, runs
 * dlrm_sparse_fwd, and copies out back to host, all ordered on `stream`.
 * bags->indices / bags->offsets and dense_host / out_host are HOST pointers
 * (pinned memory lets the copies run asynchronously); indices_dev,
 * offsets_dev, dense_dev and out_dev are device staging buffers of the same
 * sizes.  The host buffers must stay valid until the stream reaches the end
 * of the call. */
dlrm_status dlrm_sparse_fwd_host(const dlrm_tables *tables, const dlrm_bags *bags,
                                 dlrm_pool_mode mode, const float *dense_host,
                                 float *out_host, void *indices_dev,
                                 void *offsets_dev, float *dense_dev,
                                 float *out_dev, int32_t *status_dev,
                                 cudaStream_t stream);

/* Bytes of device workspace dlrm_sparse_bwd_adagrad needs for these shapes. */
dlrm_status dlrm_sparse_bwd_workspace_size(const dlrm_tables *tables,
                                           const dlrm_bags *bags,
                                           size_t *bytes);

/* One training step of the sparse path (fp32 tables only):
 *   1. interaction backward: with g(i,j) = g(j,i) = grad_out[b][D + pos(i,j)],
 *      dV_i = sum_{j != i} g(i,j) V_j;  grad_dense = grad_out[b][0:D] + dV_0;
 *      dP[b][t] = dV_{1+t}   (V rebuilt from dense and pooled_saved);
 *   2. per embedding row r, g_r = sum of dP[b][t] (times 1/L in mean mode)
 *      over the lookups of r, reduced in lookup order after a stable radix
 *      sort of the lookups by row (bitwise reproducible run to run);
 *   3. row-wise Adagrad on every touched row, in place:
 *      A_r += mean_d(g_r,d^2);  w_r,d -= lr * g_r,d / (sqrt(A_r) + eps).
 *      Rows not looked up are not touched.
 * tables: the same tables as the forward, updated in place (dtype must be
 * DLRM_F32).  accum: HOST array of T device pointers, accumulator of table t
 * has V_t fp32 entries, updated in place.  dense, pooled_saved (device,
 * B x T x D from dlrm_sparse_fwd), grad_out (device, B x (D+N(N-1)/2)),
 * grad_dense (device, B x D, written).  workspace: device, at least
 * dlrm_sparse_bwd_workspace_size() bytes, 16-byte aligned, contents ignored.
 * Ordering: the step is one operation on `stream`, after the work queued on
 * it before the call and before the work queued after.  side_stream is
 * optional: NULL (or equal to stream) runs every kernel on `stream`; another
 * stream of the same device takes the lookup-key build and the sort of
 * step 2, which then run beside step 1.  That stream is forked from `stream`
 * and joined back to it by two events the call creates and releases (no
 * state outlives the call), so the caller may reuse it for anything else and
 * the pattern holds under stream capture.  The library keeps no global
 * state: calls on different streams are independent.
 * Limits (DLRM_ERR_UNSUPPORTED): total rows over all tables < 2^32 - 1,
 * T * B < 2^32, nnz < 2^32 (32-bit sort keys, values and positions). */
dlrm_status dlrm_sparse_bwd_adagrad(const dlrm_tables *tables, const dlrm_bags *bags,
                                    dlrm_pool_mode mode, const float *dense,
                                    const float *pooled_saved,
                                    const float *grad_out, float *grad_dense,
                                    float *const *accum, float lr, float eps,
                                    void *workspace, size_t workspace_bytes,
                                    int32_t *status_dev, cudaStream_t stream,
                                    cudaStream_t side_stream);

/* Bytes of the fixed scratch behind dlrm_sparse_bwd_adagrad_static. */
#define DLRM_STATIC_SCRATCH_BYTES (32u << 20)

/* dlrm_sparse_bwd_adagrad for callers that cannot allocate device memory
 * (the pages have no counterpart: this is a library convenience).  Such
 * callers are, for example, a plugin reached through a plain C interface
 * that receives only its input and output buffers, or a process whose device
 * memory is owned by another framework's pooled allocator.  Instead of a
 * caller workspace the step uses one fixed array of
 * DLRM_STATIC_SCRATCH_BYTES of device memory that the library holds on every
 * device that loads it, until the process exits.  Arguments, layouts and
 * results are those of dlrm_sparse_bwd_adagrad without workspace /
 * workspace_bytes and side_stream (every kernel runs on `stream`).
 *   - Returns DLRM_ERR_INVALID_ARG, before touching the GPU, when the batch
 *     needs more scratch than DLRM_STATIC_SCRATCH_BYTES
 *     (dlrm_sparse_bwd_workspace_size() says how much it needs).
 *   - Every call looks up the array's device address on the current device
 *     (the first call on a device also loads that part of the library onto
 *     it); make that first call before any stream capture.  Looking it up
 *     each time keeps the address right after the device's context has been
 *     reset and made again.
 *   - All calls on a device share the array: calls that overlap on the GPU
 *     (other streams, or host threads without ordering) race and must be
 *     serialised by the caller.  No scratch contents carry over between
 *     calls; nothing needs clearing.
 *   - Allocates nothing: no cudaMalloc, no cudaFree. */
dlrm_status dlrm_sparse_bwd_adagrad_static(const dlrm_tables *tables, const dlrm_bags *bags,
                                           dlrm_pool_mode mode, const float *dense,
                                           const float *pooled_saved,
                                           const float *grad_out, float *grad_dense,
                                           float *const *accum, float lr, float eps,
                                           int32_t *status_dev, cudaStream_t stream);

/* A static, human-readable name of the lowest set status bit. */
const char *dlrm_status_string(dlrm_status status);

/* Version of this ABI (bumped when a signature or layout changes). */
int32_t dlrm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DLRM_SPARSE_H */
