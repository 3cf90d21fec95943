// plan.cuh -- the plan handle: copied column descriptors, device metadata and
// the workspace sized once at creation (library-internal).
#pragma once

#include <vector>

#include "common.cuh"

namespace emb {

// Forward: threads per CTA (each warp works alone on its tiles); bags longer
// than kLongBag values are pooled by the whole warp; a tile covers at most
// kMaxTileElems stream elements (bags are owned by the tile that holds their
// first element).
constexpr int kFwdThreads = 256;
constexpr int kLongBag = 128;
constexpr int kMaxTileElems = 8192;

// Backward: the run-reduction CTAs take at least this many sorted entries
// each; the per-CTA partial buffers are sized for n / kUnit CTAs.
constexpr int kUnit = 128;
constexpr uint32_t kPadBit = 0x80000000u;

// Radix sort geometry (LSD, chained scan with decoupled look-back): threads
// per CTA and 32-bit pairs per thread of a tile.
constexpr int kSortThreads = 512;
constexpr int kSortItems = 15;
constexpr int kSortTile = kSortThreads * kSortItems;

struct Workspace {
  // sort buffers: keys (global rows) and values (gradient sources)
  uint32_t* keys[2] = {nullptr, nullptr};
  uint32_t* vals[2] = {nullptr, nullptr};
  float* inv_n = nullptr;          // [n_cols * max_batch] 1/n_valid of mean bags
  uint2* rec_src = nullptr;        // [max_ids] weighted forwards: (gradient source, weight bits) per record
  uint32_t* hist = nullptr;        // the sort's scratch: histograms, tile tickets, look-back words
  uint32_t* run_head = nullptr;    // [max_ids + 1] debug: runs started at or before each position
  uint32_t* head_pos = nullptr;    // [max_ids] debug: position of each run's first entry
  uint32_t* n_runs = nullptr;      // [1]
  uint32_t* scan_part = nullptr;   // per-block partial counts for run compaction
  float4* partial = nullptr;       // [n_units][2][max_dim/4] cut-run partial sums
  int32_t* part_pos = nullptr;     // [n_units][2] run boundaries of those partials
  uint8_t* part_thru = nullptr;    // [n_units] CTA lies inside one continuing run
  // atomic backward (EMB_PLAN_ATOMIC_BACKWARD)
  uint32_t* touched = nullptr;     // [ceil(rows / 32)] bitmap of the rows a step touches (kept clear)
  uint32_t* bit_part = nullptr;    // per 1024-word block: set bits, then their exclusive prefix
  int64_t* n_uniq = nullptr;       // [1] touched rows of the step
  uint32_t* uniq = nullptr;        // [max_ids] touched global rows, ascending (slot -> row)
  uint32_t* slot_of = nullptr;     // [rows] global row -> slot, valid for the step's touched rows
  float* cgrad = nullptr;          // [max_ids, max_dim] compact gradient (kept zero between steps)
  uint32_t* ucount = nullptr;      // [max_ids] debug: contributions per slot (kept zero)
  int64_t max_tiles = 0;
  int64_t n_units_max = 0;
  size_t bytes = 0;
};

}  // namespace emb

struct emb_plan_s {
  int32_t n_cols = 0;
  int32_t max_batch = 0;
  int64_t max_ids = 0;
  uint32_t flags = 0;
  bool training = false;
  bool atomic_bwd = false;             // backward by atomics into a compact gradient
  std::vector<emb_column_desc> cols;
  std::vector<emb::ColMeta> meta_h;
  std::vector<int32_t> col_table;
  std::vector<emb::TableMeta> tables_h;
  std::vector<int32_t> table_first_col;   // first column of each table
  bool low_precision = false;            // some table is stored below fp32
  std::vector<uint32_t> table_base_h;  // [n_tables + 1]
  emb::ColMeta* meta_d = nullptr;      // id-stream columns, then f-stream columns, in plan order
  int4* colg_d = nullptr;              // per column: (out_col, 1 if MEAN, dim/4) for the backward
  emb::TableMeta* tables_d = nullptr;
  uint32_t* table_base_d = nullptr;
  int32_t n_stream_cols[2] = {0, 0};
  int32_t n_tables = 0;
  int32_t n_padded = 0;
  int32_t max_dim = 0;
  int64_t out_width = 0;
  int64_t seq_per_bag = 0;
  uint32_t key_total = 0;              // sum of table rows == sentinel key
  int key_bits = 0;
  uint32_t* status_d = nullptr;
  unsigned long long* fwd_ticket = nullptr;   // forward tile tickets (next tile, warps done)
  int32_t* col_order_d = nullptr;   // per stream: its columns' stream positions, widest stored rows first
  // Padded columns with pad_len > kLongBag: the forward copies their bags in
  // pieces of positions, dealt as tiles of their own.
  int32_t n_long_padded = 0;
  int32_t max_long_pad = 0;
  bool long_padded_only[2] = {false, false};   // per stream: it has columns, all long padded
  int32_t* pad_cols_d = nullptr;               // their positions in meta_d
  int sm_count = 0;
  int fwd_ctas_per_sm = 0;
  emb::Workspace ws;
  // what the last forward recorded for the backward
  bool have_forward = false;
  int32_t last_batch = 0;
  int64_t last_n = 0;
  int64_t last_n_ids = 0;
  bool last_weighted = false;   // the last forward carried value weights (records hold rec_src)
};

namespace emb {

inline emb_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return EMB_OK;
  if (e == cudaErrorMemoryAllocation) return EMB_ERR_OOM;
  return EMB_ERR_CUDA;
}

#define EMB_CUDA_TRY(x)                                  \
  do {                                                   \
    cudaError_t _e = (x);                                \
    if (_e != cudaSuccess) return ::emb::cuda_status(_e); \
  } while (0)

// Device memory of the plan and hash handles: every allocation goes through
// dev_alloc and every release through dev_free (plan.cu), which keep a count
// of live allocations and can be armed to fail one allocation on the host
// (emb_debug_fail_alloc), so that tests reach each error path of a create
// call without exhausting the GPU.  dev_free(nullptr) does nothing.
cudaError_t dev_alloc(void** p, size_t bytes);
void dev_free(void* p);

// Launch-side entry points implemented in forward.cu / backward.cu / atomic.cu.
emb_status launch_forward(emb_plan_s* p, int32_t batch, const int64_t* ids, const int32_t* id_offsets,
                          const float* id_weights, int64_t n_ids, const float* fvals, const int32_t* f_offsets,
                          const float* f_weights, int64_t n_fvals, float* out, float* seq_out, int64_t* rows_dbg,
                          cudaStream_t stream);
int forward_ctas_per_sm();

emb_status launch_backward(emb_plan_s* p, const float* grad_out, const float* grad_seq,
                           float lr, float eps, cudaStream_t stream,
                           const emb_backward_debug* dbg);
emb_status launch_backward_atomic(emb_plan_s* p, const float* grad_out, const float* grad_seq, float lr, float eps,
                                  cudaStream_t stream, const emb_backward_debug* dbg);

}  // namespace emb
