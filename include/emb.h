/*
 * emb.h -- C ABI of the GB300 multi-column embedding front end
 * (libsparse_lookup.so, sparse_lookup_gb300/csrc).
 *
 * One process, one GPU (sm_103a).  Plain pointers and sizes only.  Unless a
 * parameter says "(host)", every pointer is a DEVICE pointer in the current
 * CUDA context.  `stream` is a cudaStream_t passed as void* (NULL = legacy
 * default stream).  All calls are stream-ordered and asynchronous unless they
 * say they synchronize.  No handle is thread-safe; use one handle per thread.
 *
 * Pages the operations follow, by title and section:
 *  [RecIS]    "RecIS: Unifying Sparse and Dense Computation for Efficient
 *             Recommendation Training": §3.1 fused feature transforms (hash,
 *             modulo, bucketize; element-count tiling; 16-byte vector access),
 *             §3.2 "Index-aware segment reduction" and Algorithm 1 (CSR
 *             forward with a unique writer per output; backward as the sum of
 *             per-contributor gradients), Figure 3 (local reduce-ID), §4.3
 *             (sparse learning rate 0.01).
 *  [RECom]    "RECom: A Compiler Approach to Accelerating Recommendation Model
 *             Inference with Massive Embedding Columns": "Why this problem is
 *             worth solving" (an embedding column = transform to an index,
 *             safety handling, lookup, reduce; thousands of columns fused in
 *             one kernel), "How RECom works" (empty-row filling merged into the
 *             lookup, range guards).
 *  [Monolith] "Di Dalam Monolit ByteDance: Mesin yang Memberdayakan Umpan
 *             Konten yang Lebih Cerdas dan Cepat": §2.1 "Tabel Hash"
 *             (collision-free key-value table, admission by occurrence count,
 *             expiry of idle IDs).
 *
 * Errors.  Argument checks are synchronous and return a status before any
 * work is queued; they leave no CUDA error pending.  Conditions only the GPU
 * can see (probe limit, full row pool, invalid offsets, a wait that ran out)
 * are latched into a device status word of the handle; read and clear it with
 * emb_get_device_status / hash_get_device_status, which synchronize `stream`.
 * Kernels never trap, assert or wait without a bound.
 */
#ifndef SPARSE_LOOKUP_EMB_H
#define SPARSE_LOOKUP_EMB_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EMB_OK = 0,
    EMB_ERR_INVALID_ARG = 1,  /* bad pointer, size, layout or value          */
    EMB_ERR_UNSUPPORTED = 2,  /* valid but outside this build's limits       */
    EMB_ERR_OOM = 3,          /* device or host allocation failed            */
    EMB_ERR_CUDA = 4,         /* a CUDA runtime call failed                  */
    EMB_ERR_TABLE_FULL = 5,   /* hash: no free row for an admitted key       */
    EMB_ERR_PROBE_LIMIT = 6,  /* hash: max_probes slots probed, no place     */
    EMB_ERR_BAD_INDEX = 7,    /* device saw offsets outside the given values */
    EMB_ERR_TIMEOUT = 8       /* a bounded device wait gave up               */
} emb_status;

/* Feature transform of a column [RecIS §3.1; RECom "Why this problem is
 * worth solving"]. */
typedef enum {
    EMB_T_IDENTITY = 0,   /* int64 value is the row                          */
    EMB_T_HASH_MOD = 1,   /* row = splitmix64((u64)value) mod num_rows:
                             one SplitMix64 output with state = value        */
    EMB_T_BUCKETIZE = 2,  /* fp32 value; row = #{j : boundaries[j] <= value};
                             NaN -> 0; num_rows = num_boundaries + 1         */
    EMB_T_ROWS_GIVEN = 3  /* int64 row produced by hash_lookup_or_insert;
                             -1 (not admitted) is dropped                    */
} emb_transform;

/* Reduction of a bag [RecIS §3.2 Algorithm 1, forward]. */
typedef enum {
    EMB_POOL_SUM = 0,         /* sum of the valid rows                        */
    EMB_POOL_MEAN = 1,        /* sum / number of valid rows                   */
    EMB_POOL_NONE_PADDED = 2  /* no pooling: rows copied to [batch, pad_len,
                                 dim], zero past the bag end and for dropped
                                 IDs; the bag is cut after pad_len values     */
} emb_pooling;

/* Storage type of a table's rows (the RecIS evaluation lists an int8 table
 * beside fp32 ones, Table 3).  Lookups convert each element to fp32 and pool
 * in fp32: bf16 and fp16 convert exactly; int8 element q of row r reads as
 * row_scale[r] * q (one fp32 rounding).  Low-precision tables are read-only:
 * only inference plans take them. */
typedef enum {
    EMB_DT_F32 = 0,
    EMB_DT_BF16 = 1,
    EMB_DT_F16 = 2,
    EMB_DT_I8 = 3
} emb_table_dtype;

/* Safety handling [RECom "Why this problem is worth solving"]: a value whose
 * row falls outside [0, num_rows) is dropped (it reads nothing, counts for
 * nothing, receives no gradient).  A pooled bag with no valid value yields
 * default_vec (zeros when NULL) and passes no gradient. */
typedef struct {
    int32_t transform;        /* emb_transform                                   */
    int32_t pooling;          /* emb_pooling                                     */
    int64_t num_rows;         /* 1 <= num_rows < 2^31                            */
    int32_t dim;              /* 4 <= dim <= 256, dim % 4 == 0                   */
    int32_t pad_len;          /* EMB_POOL_NONE_PADDED: >= 1; otherwise ignored   */
    const float* boundaries;  /* EMB_T_BUCKETIZE: [num_boundaries] fp32, strictly
                                 increasing, 1 <= num_boundaries <= 4096         */
    int32_t num_boundaries;
    int32_t max_len;          /* EMB_POOL_SUM / MEAN: pool only the first max_len
                                 values of each bag, the rest read nothing and get
                                 no gradient (sequence truncation, RecIS §2.1);
                                 0 = all.  Must be 0 for EMB_POOL_NONE_PADDED
                                 (pad_len cuts there).                          */
    float* weight;            /* [num_rows, dim] row-major in table_dtype (fp32
                                 unless stated), 16-byte aligned.  Columns given
                                 the SAME pointer share one table (same
                                 num_rows, dim and table_dtype required); the
                                 backward then merges their gradients per row. */
    float* adagrad_acc;       /* [num_rows, dim] fp32 Adagrad accumulator, same
                                 sharing; required by training plans             */
    const float* default_vec; /* [dim] fp32 or NULL (zeros)                      */
    int32_t table_dtype;      /* emb_table_dtype; 0 = fp32                       */
    int32_t reserved;         /* 0                                               */
    const float* row_scale;   /* EMB_DT_I8: [num_rows] fp32 scale per row,
                                 4-byte aligned; otherwise ignored               */
} emb_column_desc;

/* Plan flags. */
#define EMB_PLAN_TRAINING 1u  /* allocate the backward workspace; emb_forward
                                 then also records what the backward needs   */
#define EMB_PLAN_ATOMIC_BACKWARD 2u
                              /* with EMB_PLAN_TRAINING: emb_backward_update
                                 merges equal rows inside each warp and adds
                                 the sums to a compact gradient with global
                                 atomics instead of sorting [RecIS §3.2
                                 Algorithm 1, backward]; extra device memory:
                                 4 B per table row (row -> slot map) plus
                                 max_ids * max_dim * 4 B (compact gradient).
                                 Same update; the summation order then depends
                                 on scheduling (results within the fp32
                                 summation bound, not bit-identical run to
                                 run).                                        */

typedef struct emb_plan_s* emb_plan;

/* emb_plan_create -- validate and copy `n_cols` column descriptors and size
 * every workspace once, so that emb_forward and emb_backward_update never
 * allocate.  The plan replaces the per-column graphs that RECom compiles into
 * one kernel [RECom "How RECom works"]: all columns run in one forward launch.
 *
 *  cols      (host) [n_cols] descriptors; copied, the caller may free them.
 *            Tables, accumulators, boundaries and defaults stay caller-owned
 *            and must outlive the plan.
 *  n_cols    1 .. 65535
 *  max_batch 1 .. 2^31-1; n_cols * max_batch < 2^31
 *  max_ids   training plans: the largest n_ids + n_fvals a forward will see
 *            (< 2^30: the backward's radix sort counts in 30 bits); ignored
 *            otherwise
 *  flags     EMB_PLAN_TRAINING or 0
 *  out       (host) receives the plan
 * Limits: the distinct tables' row counts must sum below 2^32 - 1 (the
 * backward sorts 32-bit global row keys).
 * Returns EMB_ERR_INVALID_ARG / EMB_ERR_UNSUPPORTED / EMB_ERR_OOM /
 * EMB_ERR_CUDA; on error *out is NULL and nothing is leaked. */
emb_status emb_plan_create(const emb_column_desc* cols, int32_t n_cols, int32_t max_batch,
                           int64_t max_ids, uint32_t flags, emb_plan* out);

/* Frees the plan's own memory (not the caller's tables).  Synchronizes the
 * device so that no queued kernel still uses the workspace. */
emb_status emb_plan_destroy(emb_plan plan);

/* emb_plan_info -- layout facts of a plan, all outputs (host) and optional:
 *  out_width          floats per row of the pooled output (sum of the pooled
 *                     columns' dims, in column order)
 *  seq_floats_per_bag floats per bag of the padded output (sum over padded
 *                     columns of pad_len * dim)
 *  n_tables           distinct tables (by weight pointer)
 *  col_table          [n_cols] table index of each column, tables numbered in
 *                     order of first appearance
 *  workspace_bytes    device bytes the plan owns */
emb_status emb_plan_info(emb_plan plan, int64_t* out_width, int64_t* seq_floats_per_bag,
                         int32_t* n_tables, int32_t* col_table, int64_t* workspace_bytes);

/* emb_forward -- transform, guard, gather and pool every column of the plan
 * in one pass [RecIS §3.1, §3.2 Algorithm 1 forward; RECom "Why this problem
 * is worth solving"].
 *
 * Inputs are two jagged (CSR) streams over (column, bag) segments, columns
 * in plan order, bags 0..batch-1 inside each column:
 *  ids, id_offsets  int64 values of the non-BUCKETIZE columns: segment
 *                   k*batch + b (k-th such column) holds
 *                   ids[id_offsets[k*batch+b] .. id_offsets[k*batch+b+1]).
 *                   id_offsets has n_id_cols*batch + 1 int32 entries,
 *                   id_offsets[0] == 0, non-decreasing, last == n_ids.
 *  fvals, f_offsets the same for the BUCKETIZE columns (fp32 values).
 *  id_weights, f_weights  optional fp32 weights, one per value of each
 *                   stream (NULL: none).  A SUM column of a weighted stream
 *                   pools sum_r w_r * E[row_r] and its backward passes
 *                   w_r * G to row_r [RecIS §3.2 Algorithm 1, w_r]; MEAN and
 *                   padded columns ignore the weights.
 *  n_ids, n_fvals   element counts of the two value arrays.  Offsets outside
 *                   [0, n] are clamped on the device (never read out of
 *                   bounds) and latch EMB_ERR_BAD_INDEX.
 * Outputs:
 *  out      [batch, out_width] fp32: pooled column c occupies floats
 *           [col_off_c, col_off_c + dim_c) of each row (columns concatenated
 *           in plan order).  16-byte aligned.  Each element has exactly one
 *           writer; no atomics.
 *  seq_out  padded columns, concatenated in plan order, each [batch, pad_len,
 *           dim] fp32; NULL if the plan has none.  16-byte aligned.
 *  rows_dbg optional [n_ids + n_fvals] int64: transformed row of every value
 *           (id stream first), -1 where dropped.  NULL in production.
 * A training plan also records, in its workspace, each contribution's row and
 * bag for emb_backward_update; batch <= max_batch and n_ids + n_fvals <=
 * max_ids are then required (the weights are copied there too, 8 B per
 * value).  The input buffers must stay unchanged until the backward of this
 * forward has been queued.
 * Calls on one plan must be ordered (one stream, or streams joined by events):
 * the forward's tile counter and the training workspace belong to the plan. */
emb_status emb_forward(emb_plan plan, int32_t batch,
                       const int64_t* ids, const int32_t* id_offsets, const float* id_weights, int64_t n_ids,
                       const float* fvals, const int32_t* f_offsets, const float* f_weights, int64_t n_fvals,
                       float* out, float* seq_out, int64_t* rows_dbg, void* stream);

/* Optional device outputs of emb_backward_update, for parity checks. */
typedef struct {
    int64_t* n_unique;   /* [1] number of distinct (table, row) touched        */
    int32_t* uniq_table; /* [max_ids] table index of each unique row, ascending
                            by (table, row)                                   */
    int64_t* uniq_row;   /* [max_ids] row inside its table                     */
    int32_t* counts;     /* [max_ids] contributions per unique row             */
    float* agg_grad;     /* [max_ids, max_dim] aggregated gradient (first dim
                            floats of each row used)                          */
} emb_backward_debug;

/* emb_backward_update -- backward of the last emb_forward on this plan plus
 * one sparse Adagrad step [RecIS §3.2 Algorithm 1 backward semantics; Figure 3
 * local reduce-ID; §4.3 sparse learning rate].
 *
 * Every valid contribution r of bag b of column c carries scale_r *
 * grad_out[b, col_off_c : col_off_c + dim_c] (scale w_r for SUM -- 1 without
 * weights --, 1/n_valid for MEAN), or grad_seq[b, t, :] of its padded column.  The contributions are
 * radix-sorted by global row, the runs give the unique rows and counts, each
 * unique row's gradient g is summed by exactly one writer (atomic plans: a
 * bitmap of touched rows gives them in ascending order and g is accumulated
 * with atomics), then
 *   acc += g*g;  w -= lr * g / (sqrt(acc) + eps)
 * element-wise in fp32 (torch.optim.Adagrad with lr_decay = weight_decay = 0).
 * Rows not touched by the batch are not read or written.
 *  grad_out  [batch, out_width] fp32 (NULL only if no pooled column)
 *  grad_seq  padded columns' gradient, laid out like seq_out (or NULL)
 *  dbg       (host) optional struct of optional device outputs, or NULL
 * Requires a training plan and a preceding emb_forward on the same stream. */
emb_status emb_backward_update(emb_plan plan, const float* grad_out, const float* grad_seq,
                               float lr, float eps, void* stream, const emb_backward_debug* dbg);

/* Synchronizes `stream`, returns the first device-side error latched since
 * the last call (EMB_OK if none) and clears it. */
emb_status emb_get_device_status(emb_plan plan, void* stream);

/* ------------------------------------------------------------------------ */
/* Collision-free dynamic table [Monolith §2.1 "Tabel Hash"]                */
/* ------------------------------------------------------------------------ */

typedef struct emb_hash_s* emb_hash;

/* hash_create -- a GPU key -> row table over a private row pool.
 *  num_slots      power of two, 2^10 .. 2^31: open-addressing slots of 16 B.
 *                 Expired entries leave tombstones; inserts reuse them and
 *                 expiry turns a tombstone run that ends at an empty slot
 *                 back into empty slots.  Keep the live keys well below
 *                 num_slots (probe lengths grow with the load).
 *  row_capacity   rows in the pool, 1 .. 2^31-1
 *  dim            floats per row (4..256, multiple of 4)
 *  admit_threshold occurrences a key needs before it gets a row (>= 1)
 *  max_probes     bound on the slots one lookup may probe (>= 1)
 *  init_seed, init_scale: a new row's element d is
 *                 init_scale * ((splitmix64(key ^ (tid << 48) ^ seed ^ d)
 *                 >> 40) - 2^23) * 2^-23, its accumulator 0.
 *  max_keys_per_call  largest n a hash_lookup_or_insert will pass (< 2^30);
 *                 sizes the admission workspace and 16 lists of touched slots
 *                 (about 95 B per key in all) so lookups never allocate.
 *  out            (host) receives the handle.
 * Keys are (table id, key) pairs with 0 <= tid < 2^15 and 0 <= key < 2^48;
 * distinct pairs never share an entry or a row.  Allocates the slots, the
 * row pool and the workspace once and synchronizes the device. */
emb_status hash_create(int64_t num_slots, int64_t row_capacity, int32_t dim,
                       int32_t admit_threshold, int32_t max_probes, uint64_t init_seed,
                       float init_scale, int64_t max_keys_per_call, emb_hash* out);

/* Borrowed views of the row pool: weight and accumulator [row_capacity, dim]
 * fp32, owned by the handle (valid until hash_destroy).  Either may be NULL. */
emb_status hash_rows(emb_hash h, float** weight, float** acc);

/* hash_lookup_or_insert -- one batch of n occurrences at `step`.
 * Every occurrence touches its entry (last_seen = step); while a key is not
 * admitted each occurrence adds 1 to its count.  After the whole batch is
 * counted, keys whose count reached admit_threshold are admitted in
 * ascending (tid, key) order, each taking the lowest free row (rows released
 * by expiry first, then never-used rows); their rows are initialised as in
 * hash_create.  rows_out[i] is the row of occurrence i, or -1 while its key
 * is not admitted (also for a key outside the key range, which latches
 * EMB_ERR_INVALID_ARG).  A full pool latches EMB_ERR_TABLE_FULL (the keys left
 * without a row keep counting and are admitted by their first occurrence in a
 * later call, once rows are free; calls are told apart by `step`, so steps of
 * consecutive calls should differ); probing max_probes slots without a place
 * latches EMB_ERR_PROBE_LIMIT and returns -1 for that occurrence.
 *  table_ids [n] int32; keys [n] int64; rows_out [n] int64 (feeds emb_forward
 *  columns of transform EMB_T_ROWS_GIVEN directly).  n <= max_keys_per_call.
 *  step      any value but 2^32 - 1 (which marks slots never touched). */
emb_status hash_lookup_or_insert(emb_hash h, const int32_t* table_ids, const int64_t* keys,
                                 int64_t n, uint32_t step, int64_t* rows_out, void* stream);

/* hash_evict_expired -- remove every entry, admitted or still counting, with
 * now - last_seen > ttl; admitted rows return to the free pool.  Each lookup
 * lists the slots it touched first; an expiry checks only the lists of steps
 * more than ttl behind `now`.  With one lookup per step and ttl <= 14 that is
 * the whole work; a second lookup at one step, or more than 16 steps with
 * live lists, makes expiries sweep every slot until those lookups are more
 * than ttl steps old.  The result is the same either way.
 * n_evicted_dev: optional device int64 receiving the number removed. */
emb_status hash_evict_expired(emb_hash h, uint32_t now, uint32_t ttl, void* stream,
                              int64_t* n_evicted_dev);

/* hash_export -- every live entry, in no particular order: tids, keys, rows
 * (-1 while counting), counts (occurrences counted so far while counting; -1
 * once admitted), last_seen; each output is an optional device array of `cap`
 * entries.  *n_out (host) receives the number of live entries (which may
 * exceed cap: only cap are written).  Synchronizes `stream`. */
emb_status hash_export(emb_hash h, int32_t* tids, int64_t* keys, int64_t* rows, int32_t* counts,
                       uint32_t* last_seen, int64_t cap, int64_t* n_out, void* stream);

/* hash_import -- restores the table from a snapshot that hash_export wrote
 * (checkpoint and resume: the pages' table is restored from snapshots of the
 * parameter servers [Monolith §2.3]).  The table is cleared first (every slot
 * empty, every row free); it then holds exactly the n entries given, with the
 * same meaning as hash_export's outputs: tids, keys, rows (the admitted
 * entry's row, -1 while counting), counts (occurrences counted while
 * counting; NULL = 0), last_seen.  Rows keep their numbers, so the row pool
 * restored through hash_rows (the caller copies the weights and accumulators
 * back) matches the entries; the pool itself is not touched.  Later lookups,
 * admissions and expiries then behave as they would have on the table the
 * snapshot was taken from.  Checked on the device: key range, distinct
 * (tid, key) pairs, admitted rows below row_capacity and distinct, counts
 * >= 0, last_seen != 2^32 - 1; a bad entry is left out and latches
 * EMB_ERR_INVALID_ARG (the table then holds the other entries, and rows a
 * rejected entry claimed may stay marked used: import a good snapshot
 * again); max_probes slots probed without a place latches
 * EMB_ERR_PROBE_LIMIT.  Expiries sweep every slot until the latest imported
 * last_seen is more than ttl behind.  All arrays device [n];
 * n <= num_slots.  Synchronizes `stream`. */
emb_status hash_import(emb_hash h, const int32_t* tids, const int64_t* keys, const int64_t* rows,
                       const int32_t* counts, const uint32_t* last_seen, int64_t n, void* stream);

/* Synchronizes `stream`, returns and clears the latched device status. */
emb_status hash_get_device_status(emb_hash h, void* stream);

/* Frees the table and its row pool (synchronizes the device first). */
emb_status hash_destroy(emb_hash h);

/* emb_sparse_adagrad_noalloc -- one sparse Adagrad step on one table, with
 * duplicate rows merged, that allocates no memory.  The pages have no
 * counterpart to this call: it exists for callers that cannot call
 * cudaMalloc -- a host framework that owns all device memory through its own
 * pool (a raw allocation would bypass its accounting or fail against its
 * reservation), a serving process that forbids allocation after start-up to
 * keep latency bounded, or a plugin that is only ever handed pointers.  Such
 * callers cannot create a plan, whose workspace is allocated at creation.
 *
 * rows[i] (int64, [n]) names the row that gradient grads[i, :] (fp32 [n, dim],
 * row-major, 16-byte aligned) belongs to; rows outside [0, num_rows) are
 * ignored.  The gradients of equal rows are summed (same sort, run reduction
 * and fp32 Adagrad as emb_backward_update), then every touched row of weight
 * and acc ([num_rows, dim] fp32, 16-byte aligned) takes one step
 *   acc += g*g;  w -= lr * g / (sqrt(acc) + eps).
 *
 * Scratch: a fixed area of about 8.6 MB compiled into the library as a
 * file-scope device array; every GPU that loads the library holds it until
 * the process exits.  Limits: n <= 262144 (2^18), dim <= 256, num_rows <
 * 2^31; larger sizes return EMB_ERR_UNSUPPORTED before any work is queued.
 * The first call on a device looks up the area's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls on a device share the one area, which keeps the last
 * call's contents (each call clears what must start at zero): calls whose
 * work overlaps on the GPU -- on different streams, or from different host
 * threads -- race and corrupt each other's results; serialize them.
 * Device-side errors (a wait of the sort that ran out: EMB_ERR_TIMEOUT) are
 * latched into a status word of the area, read and cleared by
 * emb_noalloc_get_device_status; a call whose sort gave up a wait leaves
 * weight and acc untouched.
 * Calls no cudaMalloc, cudaFree or allocating library routine. */
emb_status emb_sparse_adagrad_noalloc(const int64_t* rows, int64_t n, const float* grads, float* weight,
                                      float* acc, int64_t num_rows, int32_t dim, float lr, float eps,
                                      void* stream);

/* emb_noalloc_get_device_status -- companion of emb_sparse_adagrad_noalloc
 * (no counterpart on the pages either): synchronizes `stream`, returns the
 * first device-side error latched by emb_sparse_adagrad_noalloc calls on the
 * current device since the last query (EMB_OK if none) and clears it.
 * Allocates nothing (the word lives in the same file-scope area). */
emb_status emb_noalloc_get_device_status(void* stream);

/* ------------------------------------------------------------------------ */
/* Self tests and fault injection (no counterpart on the pages)              */
/* ------------------------------------------------------------------------ */

/* emb_selftest_sort_timeout -- makes the bounded wait of the radix sort's
 * decoupled look-back run out on purpose, without faulting or hanging the
 * GPU: one pass over two tiles in which only the second tile runs, so its
 * wait for the first tile's counts can never end; after its bound (about a
 * second) the tile latches EMB_ERR_TIMEOUT and raises the sort's fail word,
 * then a run reduction over the incomplete output must see that word and
 * leave its table untouched.  Allocates and frees its own small buffers and
 * synchronizes the device.  All pointers are host:
 *  latched          the status the sort latched (EMB_ERR_TIMEOUT expected)
 *  fail_word        the sort's fail word afterwards (nonzero expected)
 *  table_untouched  1 if the reduction left its table as it was
 *  wait_ms          optional: device time of the waiting pass */
emb_status emb_selftest_sort_timeout(uint32_t* latched, uint32_t* fail_word, int32_t* table_untouched,
                                     float* wait_ms);

/* emb_debug_fail_alloc -- host-side fault injection for the create calls:
 * after `after` more device allocations by emb_plan_create / hash_create /
 * the self tests succeed, the next one fails as if the device were out of
 * memory (nothing is asked of the driver), then the hook disarms itself.
 * after = -1 disarms it.  Every create call must then return EMB_ERR_OOM
 * with *out NULL and nothing leaked. */
emb_status emb_debug_fail_alloc(int64_t after);

/* emb_debug_live_allocations -- number and bytes (host, optional) of the
 * device allocations the library's handles hold right now. */
emb_status emb_debug_live_allocations(int64_t* count, int64_t* bytes);

/* Host-side self test of arithmetic shared by host and device code: */

/* Row of each value under a HASH_MOD column with `num_rows` rows, computed on
 * the HOST by the same inline code the kernels run (splitmix64 and the
 * division-by-invariant-integer of the modulo).  All pointers are host. */
emb_status emb_selftest_hash_mod(const int64_t* ids, int64_t n, int64_t num_rows, int64_t* rows_out);

/* emb_calibrate_gather -- measurement support, no counterpart on the pages:
 * reads rows row_idx[0..n) of table [num_rows, dim] (fp32, 16-byte aligned)
 * with the forward's access shape and nothing else, so that a benchmark can
 * time the random-row gather rate of this GPU for a row size.  row_idx are
 * uint32 rows < num_rows (not checked: the caller draws them in range); sink
 * is a device float that is practically never written. */
emb_status emb_calibrate_gather(const float* table, int64_t num_rows, int32_t dim, const uint32_t* row_idx,
                                int64_t n, float* sink, void* stream);

/* Library version string (host, static storage). */
const char* emb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_LOOKUP_EMB_H */
