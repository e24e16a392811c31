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
    DLRM_ERR_UNSUPPORTED = 32, /* valid request the library does not implement */
    DLRM_ERR_CAPACITY = 64     /* device: a staging area ran out of rows (those lookups pool as zero) */
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
 * entries) and offsets (device, T*B+1 entries) share index_type.  The
 * forward entry points take nnz <= 2^31 - 1 (DLRM_ERR_UNSUPPORTED above it;
 * int32 indices imply it), the training step nnz < 2^32. */
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
 * B x T x D or NULL (written when given, for the training step).  With
 * pooled_save given, bags of more than 1.25 lookups on average are pooled by
 * the lookup kernel into pooled_save and the interaction reads them back (two
 * kernels, the same values), which is faster for such bags than pooling on
 * chip; an inference caller with the memory to spare may pass a scratch
 * buffer here for that reason. */
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

/* Update rules of the embedding rows ("DLRM", robocikowo.com, "Forward
 * pass", last sentence: training with SGD or Adagrad).  Both act on g_r, the
 * sum over the step's lookups of row r of the gradient of the pooled vector
 * of the lookup's bag (times 1/L in mean mode), once per touched row:
 *   DLRM_RULE_ADAGRAD  row-wise Adagrad: A_r += mean_d(g_r,d^2);
 *                      w_r,d -= lr * g_r,d / (sqrt(A_r) + eps)
 *   DLRM_RULE_SGD      plain SGD: w_r,d -= lr * g_r,d (no momentum, no decay)
 * Rows that no lookup of the batch touches are left unchanged. */
typedef enum { DLRM_RULE_ADAGRAD = 0, DLRM_RULE_SGD = 1 } dlrm_update_rule;

typedef struct {
    int32_t rule;               /* dlrm_update_rule */
    float lr;                   /* learning rate */
    float eps;                  /* Adagrad: added to sqrt(A_r) */
    float *const *accum;        /* Adagrad: HOST array of T device pointers, V_t fp32
                                 * accumulators each, updated in place; SGD: unused */
} dlrm_update;

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

/* The training step of dlrm_sparse_bwd_adagrad with either update rule
 * (update->rule; update->accum only for Adagrad).  Arguments, workspace
 * (dlrm_sparse_bwd_workspace_size), streams, limits and errors as there;
 * DLRM_ERR_INVALID_ARG for an unknown rule or Adagrad without accumulators. */
dlrm_status dlrm_sparse_bwd_update(const dlrm_tables *tables, const dlrm_bags *bags,
                                   dlrm_pool_mode mode, const float *dense,
                                   const float *pooled_saved, const float *grad_out,
                                   float *grad_dense, const dlrm_update *update,
                                   void *workspace, size_t workspace_bytes,
                                   int32_t *status_dev, cudaStream_t stream,
                                   cudaStream_t side_stream);

/* The training step in two calls, so that the sort of step 2 can run while
 * the forward runs (same page and passage as dlrm_sparse_bwd_adagrad: the
 * sort depends only on the bags, which the forward already has).
 *
 * dlrm_sparse_bwd_sort builds the lookup keys (global row id, dP row) of the
 * bags and sorts them stably by row into `workspace` (at least
 * dlrm_sparse_bwd_workspace_size() bytes, 16-byte aligned), on `stream`.  It
 * reads only the bags and the tables' row counts (the tables' device memory
 * is not read; dtype must be DLRM_F32); out-of-range indices and malformed
 * offsets are flagged in status_dev as in the forward.
 *
 * dlrm_sparse_bwd_update_sorted is dlrm_sparse_bwd_update (arguments, limits,
 * errors, results bit for bit) minus the key build and the sort: it reads the
 * sorted lookups that dlrm_sparse_bwd_sort left in the same workspace.
 * sorted: optional event, recorded on the sort's stream after the sort and
 * before this call; the call queues the interaction backward (which does not
 * read the sorted lookups), then makes `stream` wait for `sorted`, then
 * queues the per-row sums.  NULL: the caller has ordered the sort before the
 * call (same stream, or its own event wait).  grad_ready: optional event the
 * call records on `stream` right after the interaction backward, so that
 * work needing only grad_dense (the bottom MLP's backward) can run on
 * another stream beside the per-row sums.  Nothing else may write the
 * workspace between the two calls (the sort writes only its key and value
 * parts, the interaction backward only the dP part, so those two may run at
 * the same time).  Bags, tables' row counts and workspace must be those of
 * the sort; other bags give wrong row updates, not an error. */
dlrm_status dlrm_sparse_bwd_sort(const dlrm_tables *tables, const dlrm_bags *bags,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t *status_dev, cudaStream_t stream);

dlrm_status dlrm_sparse_bwd_update_sorted(const dlrm_tables *tables, const dlrm_bags *bags,
                                          dlrm_pool_mode mode, const float *dense,
                                          const float *pooled_saved, const float *grad_out,
                                          float *grad_dense, const dlrm_update *update,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t *status_dev, cudaEvent_t sorted,
                                          cudaEvent_t grad_ready, cudaStream_t stream);

/* The interaction backward alone (calculus on "DLRM", robocikowo.com,
 * "Forward pass" steps (3)-(4)): with g(i,j) = g(j,i) = grad_out[b][D + pos(i,j)],
 *   dV_i = sum_{j != i} g(i,j) V_j,  grad_dense = grad_out[b][0:D] + dV_0,
 *   grad_pooled[b][t] = dV_{1+t}   (the gradient of the pooled vector itself:
 *                                   no bag length is applied here).
 * dense: device B x D; pooled: device B x T x D; grad_out: device
 * B x (D + N(N-1)/2); grad_dense: device B x D and grad_pooled: device
 * B x T x D, written.  fp32 throughout; batch = B >= 1, num_tables = T in
 * [1, DLRM_MAX_TABLES], dim = D as for the tables.  Together with
 * dlrm_embbag_bwd_update it is the training step split at the pooled vectors,
 * the point where a model-parallel step exchanges them between devices. */
dlrm_status dlrm_interact_bwd(const float *dense, const float *pooled, const float *grad_out,
                              int64_t batch, int32_t num_tables, int32_t dim,
                              float *grad_dense, float *grad_pooled, cudaStream_t stream);

/* Bytes of device workspace dlrm_embbag_bwd_update needs for these shapes
 * (mean pooling needs a scaled copy of grad_pooled). */
dlrm_status dlrm_embbag_bwd_workspace_size(const dlrm_tables *tables, const dlrm_bags *bags,
                                           dlrm_pool_mode mode, size_t *bytes);

/* Steps 2-3 of the training step from a given gradient of the pooled
 * vectors: per touched row r, g_r = sum of grad_pooled[b][t] (times 1/L in
 * mean mode) over the lookups of r, reduced in lookup order after a stable
 * radix sort by row (bitwise reproducible run to run), then one update of
 * the row by update->rule, in place.  tables (fp32, updated in place) and bags
 * as for the forward; grad_pooled: device B x T x D fp32, 16-byte aligned.
 * workspace: device, >= dlrm_embbag_bwd_workspace_size() bytes.  Streams,
 * limits and errors as for dlrm_sparse_bwd_adagrad. */
dlrm_status dlrm_embbag_bwd_update(const dlrm_tables *tables, const dlrm_bags *bags,
                                   dlrm_pool_mode mode, const float *grad_pooled,
                                   const dlrm_update *update, void *workspace,
                                   size_t workspace_bytes, int32_t *status_dev,
                                   cudaStream_t stream, cudaStream_t side_stream);

/* The raw-ID hashing pre-pass ("Deep Learning Recommendation Model (DLRM)",
 * notes.helloworld.co.in, "Why it is mostly a systems problem": IDs hashed
 * into tables of a fixed number of rows), in its plainest form, a modulo:
 *   rows[p] = raw_ids[p] mod V_t   (raw_ids read as unsigned 64-bit),
 * t the table whose bags hold position p: the last t with
 * offsets[t*B] <= p.  num_rows: HOST array of T values V_t >= 1 (at most
 * 2^31 for DLRM_I32 output).  raw_ids: device, nnz entries; offsets: device,
 * T*B+1 table-major CSR offsets of index_type; rows: device, nnz entries of
 * index_type, written (ready to serve as the bags' indices).  A position in
 * no table's range, or table boundaries that go backwards, set
 * DLRM_ERR_BAD_OFFSETS in *status_dev (such a position gets row 0). */
dlrm_status dlrm_hash_indices(const int64_t *num_rows, int32_t num_tables, int64_t batch,
                              int64_t nnz, const uint64_t *raw_ids, const void *offsets,
                              int32_t index_type, void *rows, int32_t *status_dev,
                              cudaStream_t stream);

/* ---- table-wise model parallelism ---------------------------------------
 * "DLRM" (robocikowo.com), hybrid-parallelism paragraph: the embedding tables
 * are split across devices (model parallel) while the MLPs run data
 * parallel, and the lookup results pass through an all-to-all before the
 * interaction layer; "DLRM explained", "How do you size compute for a
 * DLRM...": tables sharded across devices, an NCCL all-to-all between them.
 *
 * A plan splits the T tables among G table shards (shard g owns T_g tables,
 * pools them for all B samples into a B x T_g x D buffer, in the order of
 * its tables' slots) and the B samples among H sample shards (shard h owns
 * samples [sample_start[h], sample_start[h+1]) and runs the interaction on a
 * (sample_start[h+1] - sample_start[h]) x T x D buffer, tables in global
 * order).  All arrays are HOST memory. */
#define DLRM_MAX_SHARDS 64

typedef struct {
    int32_t num_table_shards;     /* G in [1, DLRM_MAX_SHARDS] */
    int32_t num_sample_shards;    /* H in [1, DLRM_MAX_SHARDS] */
    int32_t num_tables;           /* T in [1, DLRM_MAX_TABLES] */
    int32_t dim;                  /* D, as for the tables */
    int64_t batch;                /* B >= 1: samples of the by-table buffers */
    const int32_t *table_shard;   /* [T]: the shard g that owns table t */
    const int32_t *table_slot;    /* [T]: t's position among the tables of its shard; the
                                   * slots of a shard are 0 .. T_g - 1, each once */
    const int64_t *sample_start;  /* [H + 1]: 0 = sample_start[0] <= ... <= sample_start[H] = B */
} dlrm_shard_plan;

/* The all-to-all of the pooled vectors between the shards of a plan, on one
 * device: every (sample b, table t) row moves between by_table[g][b][slot(t)]
 * (g the owner of t) and by_sample[h][b - sample_start[h]][t] (h the sample
 * shard of b).  to_sample = 1 copies by_table -> by_sample (the forward:
 * pooled vectors to the interaction); to_sample = 0 copies by_sample ->
 * by_table (the backward: gradients of the pooled vectors back to the
 * table owners).  by_table, by_sample: HOST arrays of G and H device
 * pointers (fp32, 16-byte aligned; NULL allowed for an empty shard); the
 * source side is read, the other written; the two must not overlap.  With
 * G = H shards held by this device the call is the whole exchange; after a
 * collective all-to-all between devices, H = 1 gives the local unpack of
 * what one device received (and to_sample = 0 the pack before the reverse
 * collective).  DLRM_ERR_INVALID_ARG for an inconsistent plan. */
dlrm_status dlrm_pooled_exchange(const dlrm_shard_plan *plan, float *const *by_table,
                                 float *const *by_sample, int32_t to_sample,
                                 cudaStream_t stream);

/* ---- tables larger than device memory ------------------------------------
 * "DLRM explained", "How do you size compute for a DLRM...": tables beyond
 * device memory live in host RAM; "DLRM", robocikowo.com, CPU-inference
 * paragraph.  Item popularity follows a power law, so a device cache of the
 * hot rows takes most lookups.  Table t keeps its V_t rows in host memory the
 * device can read (pinned and mapped: cudaHostAlloc, or cudaHostRegister with
 * cudaHostRegisterMapped; on systems with unified addressing every pinned
 * allocation is), and in device memory a buffer of C_t + M_t rows: C_t cache
 * slots, then M_t staging rows for a batch's misses; plus the map slot_of (the
 * cache slot of each row, or -1) and its inverse slot_row (the row in each
 * slot, or -1).  Forward only: a training step updates rows in device memory. */
typedef struct {
    int32_t num_tables;           /* T in [1, DLRM_MAX_TABLES] */
    int32_t dim;                  /* D, as for dlrm_tables */
    int32_t dtype;                /* dlrm_dtype */
    const void *const *host_data; /* [T]: device-readable address of table t in host memory, V_t x D */
    const int64_t *num_rows;      /* [T]: V_t >= 1 */
    int32_t *const *slot_of;      /* [T]: device, V_t int32 */
    int64_t *const *slot_row;     /* [T]: device, C_t int64 */
    void *const *cache;           /* [T]: device, (C_t + M_t) x D elements, 16-byte aligned */
    const int64_t *cache_rows;    /* [T]: C_t >= 0, < 2^31 */
    const int64_t *stage_rows;    /* [T]: M_t >= 0, C_t + M_t < 2^31 */
} dlrm_tiered_tables;               /* every array above is a HOST array */

/* Empty every cache: slot_of = -1 and slot_row = -1 for every table.  Call
 * once after allocating the maps, before any other tier call. */
dlrm_status dlrm_tier_init(const dlrm_tiered_tables *tables, cudaStream_t stream);

/* Make `rows` (device, n distinct row ids of table `table`, n <= C_t) the
 * cache of that table: the rows leaving it get slot -1, rows[i] is copied from
 * host memory into slot i, slots past n hold nothing.  A row id outside
 * [0, V_t) sets DLRM_ERR_INDEX_OOB and leaves its slot empty.  Ordered on
 * `stream` like every call: no batch staged before it sees the new cache, every
 * batch staged after it does. */
dlrm_status dlrm_tier_cache_fill(const dlrm_tiered_tables *tables, int32_t table,
                                 const int64_t *rows, int64_t n, int32_t *status_dev,
                                 cudaStream_t stream);

/* Stage one batch: indices_out[p] (device, nnz entries of bags->index_type)
 * becomes the row of lookup p in the device buffer of its table: its cache
 * slot when cached, else the next staging row, into which the row is copied
 * from host memory (duplicate misses get a row each); an index outside
 * [0, V_t) becomes -1.  counters: device, T int32 of scratch (zeroed by the
 * call).  When a table's M_t staging rows run out, DLRM_ERR_CAPACITY is set in
 * *status_dev and the remaining misses become -1.  The forward entry points
 * then run on tables {cache[t], C_t + M_t rows} with these indices and the same
 * offsets, and give the result of the untiered tables bit for bit.  The
 * staging rows belong to this batch until the forward that reads them has run
 * on the stream. */
dlrm_status dlrm_tier_stage(const dlrm_tiered_tables *tables, const dlrm_bags *bags,
                            void *indices_out, int32_t *counters, int32_t *status_dev,
                            cudaStream_t stream);

/* ---- the dense layers around the sparse path ------------------------------
 * "DLRM", robocikowo.com, "Forward pass" step (1) (bottom MLP: FC layers
 * with ReLU ending at width D), step (4) and the top-MLP paragraph (FC layers
 * with ReLU, a sigmoid output), training with SGD; the hardware paragraph:
 * the MLPs are ordinary GEMMs on the tensor cores.  fp32 in and out; the
 * products run on the tcgen05 tensor cores with each fp32 operand split into
 * two bf16 values (hi + lo; hi*hi + hi*lo + lo*hi accumulated in fp32), which
 * keeps about 16 significant bits of every product (relative error below
 * 2^-16 of sum |a_k b_k|).  The split copies go to the caller's workspace;
 * the tensor cores read them through TMA tile loads.  All matrices row-major, device memory, 16-byte
 * aligned; W is out_dim x in_dim (y = x W^T + b). */
typedef enum { DLRM_ACT_NONE = 0, DLRM_ACT_RELU = 1 } dlrm_activation;

/* Bytes of device workspace dlrm_fc_fwd needs (bf16 hi / lo copies of x and W). */
dlrm_status dlrm_fc_fwd_workspace_size(int64_t batch, int32_t in_dim, int32_t out_dim, size_t *bytes);

/* y[batch][out_dim] = act(x[batch][in_dim] W^T + b); b may be NULL (no bias).
 * in_dim, out_dim in [1, 65536], batch in [1, 2^31 - 1].  workspace: device,
 * at least dlrm_fc_fwd_workspace_size() bytes, 16-byte aligned. */
dlrm_status dlrm_fc_fwd(const float *x, const float *w, const float *b, int64_t batch,
                        int32_t in_dim, int32_t out_dim, int32_t act, float *y,
                        void *workspace, size_t workspace_bytes, int32_t *status_dev,
                        cudaStream_t stream);

/* Bytes of device workspace dlrm_fc_bwd_sgd needs. */
dlrm_status dlrm_fc_bwd_workspace_size(int64_t batch, int32_t in_dim, int32_t out_dim, size_t *bytes);

/* The backward of dlrm_fc_fwd from dy (the gradient of y) with plain SGD:
 *   dz = dy * [y > 0] (act = RELU; y is the forward's output) or dy;
 *   dx = dz W  (written when dx is not NULL, with W before its update);
 *   W -= lr * dz^T x;  b -= lr * sum over the batch of dz  (when b is not NULL).
 * The sums over the batch run in a fixed order: bitwise reproducible. */
dlrm_status dlrm_fc_bwd_sgd(const float *x, float *w, float *b, const float *y, const float *dy,
                            int64_t batch, int32_t in_dim, int32_t out_dim, int32_t act,
                            float lr, float *dx, void *workspace, size_t workspace_bytes,
                            int32_t *status_dev, cudaStream_t stream);

/* Bytes of device workspace dlrm_head_bce_sgd needs (in_dim <= 1024). */
dlrm_status dlrm_head_bce_workspace_size(int64_t batch, int32_t in_dim, size_t *bytes);

/* The output layer and the loss, forward and backward with SGD: per sample
 * z = h . w + b, p = sigmoid(z) (written to prob when not NULL), the mean
 * binary cross-entropy over the batch max(z,0) - z*label + log(1+exp(-|z|))
 * (written to *loss, a device float, when not NULL); dz = (p - label) / batch;
 * dh = dz * w (written, with w before its update); w -= lr * sum dz h,
 * b -= lr * sum dz (b: one device float).  h: batch x in_dim; label: batch
 * values (0 or 1, any value in [0, 1] accepted). */
dlrm_status dlrm_head_bce_sgd(const float *h, float *w, float *b, const float *label, int64_t batch,
                              int32_t in_dim, float lr, float *prob, float *loss, float *dh,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream);

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
