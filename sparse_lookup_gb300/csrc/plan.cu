// plan.cu -- emb_plan_create / destroy / info / device status and the C-ABI
// wrappers of the forward and backward launches.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <unordered_map>

#include "plan.cuh"
#include "radix.cuh"

using namespace emb;

namespace {

std::mutex g_alloc_mu;
std::unordered_map<void*, size_t> g_live;     // live handle allocations -> bytes
int64_t g_live_bytes = 0;
std::atomic<int64_t> g_fail_after{-1};        // allocations to grant before one fails; -1 = off

}  // namespace

namespace emb {

cudaError_t dev_alloc(void** p, size_t bytes) {
  *p = nullptr;
  int64_t k = g_fail_after.load();
  while (k >= 0) {
    if (g_fail_after.compare_exchange_weak(k, k - 1)) {
      if (k == 0) return cudaErrorMemoryAllocation;   // injected: nothing was asked of the driver
      break;
    }
  }
  const cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    *p = nullptr;
    return e;
  }
  std::lock_guard<std::mutex> lk(g_alloc_mu);
  g_live[*p] = bytes;
  g_live_bytes += (int64_t)bytes;
  return cudaSuccess;
}

void dev_free(void* p) {
  if (!p) return;
  {
    std::lock_guard<std::mutex> lk(g_alloc_mu);
    auto it = g_live.find(p);
    if (it != g_live.end()) {
      g_live_bytes -= (int64_t)it->second;
      g_live.erase(it);
    }
  }
  cudaFree(p);
}

}  // namespace emb

extern "C" emb_status emb_debug_fail_alloc(int64_t after) {
  if (after < -1) return EMB_ERR_INVALID_ARG;
  g_fail_after.store(after);
  return EMB_OK;
}

extern "C" emb_status emb_debug_live_allocations(int64_t* count, int64_t* bytes) {
  std::lock_guard<std::mutex> lk(g_alloc_mu);
  if (count) *count = (int64_t)g_live.size();
  if (bytes) *bytes = g_live_bytes;
  return EMB_OK;
}

namespace {

void free_plan(emb_plan_s* p) {
  if (!p) return;
  dev_free(p->meta_d);
  dev_free(p->colg_d);
  dev_free(p->tables_d);
  dev_free(p->table_base_d);
  dev_free(p->status_d);
  dev_free(p->fwd_ticket);
  dev_free(p->col_order_d);
  dev_free(p->pad_cols_d);
  Workspace& w = p->ws;
  dev_free(w.keys[0]);
  dev_free(w.keys[1]);
  dev_free(w.vals[0]);
  dev_free(w.vals[1]);
  dev_free(w.inv_n);
  dev_free(w.rec_src);
  dev_free(w.touched);
  dev_free(w.bit_part);
  dev_free(w.n_uniq);
  dev_free(w.uniq);
  dev_free(w.slot_of);
  dev_free(w.cgrad);
  dev_free(w.ucount);
  dev_free(w.hist);
  dev_free(w.run_head);
  dev_free(w.head_pos);
  dev_free(w.n_runs);
  dev_free(w.scan_part);
  dev_free(w.partial);
  dev_free(w.part_pos);
  dev_free(w.part_thru);
  delete p;
}

template <class T>
cudaError_t dmalloc(T** ptr, size_t count, size_t* total) {
  size_t bytes = sizeof(T) * (count > 0 ? count : 1);
  *total += bytes;
  return dev_alloc((void**)ptr, bytes);
}

emb_status validate_column(const emb_column_desc& c, bool training) {
  if (c.transform < EMB_T_IDENTITY || c.transform > EMB_T_ROWS_GIVEN) return EMB_ERR_INVALID_ARG;
  if (c.pooling < EMB_POOL_SUM || c.pooling > EMB_POOL_NONE_PADDED) return EMB_ERR_INVALID_ARG;
  if (c.num_rows < 1) return EMB_ERR_INVALID_ARG;
  if (c.num_rows >= (int64_t(1) << 31)) return EMB_ERR_UNSUPPORTED;
  if (c.dim < 4 || c.dim % 4 != 0) return EMB_ERR_INVALID_ARG;
  if (c.dim > 256) return EMB_ERR_UNSUPPORTED;
  if (c.max_len < 0 || (c.pooling == EMB_POOL_NONE_PADDED && c.max_len != 0)) return EMB_ERR_INVALID_ARG;
  if (!c.weight || !aligned16(c.weight)) return EMB_ERR_INVALID_ARG;
  if (c.pooling == EMB_POOL_NONE_PADDED && c.pad_len < 1) return EMB_ERR_INVALID_ARG;
  if (c.transform == EMB_T_BUCKETIZE) {
    if (!c.boundaries || c.num_boundaries < 1) return EMB_ERR_INVALID_ARG;
    if (c.num_boundaries > 4096) return EMB_ERR_UNSUPPORTED;
    if (c.num_rows != (int64_t)c.num_boundaries + 1) return EMB_ERR_INVALID_ARG;
  }
  if (training && (!c.adagrad_acc || !aligned16(c.adagrad_acc))) return EMB_ERR_INVALID_ARG;
  if (c.default_vec && !aligned16(c.default_vec)) return EMB_ERR_INVALID_ARG;
  if (c.table_dtype < EMB_DT_F32 || c.table_dtype > EMB_DT_I8 || c.reserved != 0) return EMB_ERR_INVALID_ARG;
  if (c.table_dtype == EMB_DT_I8 && (!c.row_scale || ((uintptr_t)c.row_scale & 3u) != 0)) return EMB_ERR_INVALID_ARG;
  if (training && c.table_dtype != EMB_DT_F32) return EMB_ERR_UNSUPPORTED;   // low-precision tables are read-only
  return EMB_OK;
}

}  // namespace

extern "C" emb_status emb_plan_create(const emb_column_desc* cols, int32_t n_cols,
                                      int32_t max_batch, int64_t max_ids, uint32_t flags,
                                      emb_plan* out) {
  if (!out) return EMB_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cols || n_cols < 1 || n_cols > 65535 || max_batch < 1) return EMB_ERR_INVALID_ARG;
  if (flags & ~(EMB_PLAN_TRAINING | EMB_PLAN_ATOMIC_BACKWARD)) return EMB_ERR_INVALID_ARG;
  const bool training = (flags & EMB_PLAN_TRAINING) != 0;
  if ((flags & EMB_PLAN_ATOMIC_BACKWARD) && !training) return EMB_ERR_INVALID_ARG;
  if ((int64_t)n_cols * max_batch >= (int64_t(1) << 31)) return EMB_ERR_UNSUPPORTED;
  if (training && (max_ids < 0 || max_ids >= (int64_t(1) << 30))) return EMB_ERR_UNSUPPORTED;
  for (int32_t c = 0; c < n_cols; ++c) {
    emb_status s = validate_column(cols[c], training);
    if (s != EMB_OK) return s;
  }

  emb_plan_s* p = new (std::nothrow) emb_plan_s();
  if (!p) return EMB_ERR_OOM;
  p->n_cols = n_cols;
  p->max_batch = max_batch;
  p->max_ids = training ? max_ids : 0;
  p->flags = flags;
  p->training = training;
  p->cols.assign(cols, cols + n_cols);

  // Tables: columns with the same weight pointer share one table.
  std::map<const float*, int32_t> table_of;
  uint64_t base = 0;
  for (int32_t c = 0; c < n_cols; ++c) {
    const emb_column_desc& d = cols[c];
    auto it = table_of.find(d.weight);
    if (it == table_of.end()) {
      int32_t t = (int32_t)p->tables_h.size();
      table_of[d.weight] = t;
      TableMeta tm{};
      tm.weight = d.weight;
      tm.acc = d.adagrad_acc;
      tm.num_rows = d.num_rows;
      tm.dim = d.dim;
      tm.dim4 = d.dim / 4;
      p->tables_h.push_back(tm);
      p->table_first_col.push_back(c);
      p->table_base_h.push_back((uint32_t)base);
      base += (uint64_t)d.num_rows;
      p->col_table.push_back(t);
    } else {
      const TableMeta& tm = p->tables_h[it->second];
      const emb_column_desc& d0 = cols[p->table_first_col[it->second]];
      if (tm.num_rows != d.num_rows || tm.dim != d.dim || tm.acc != d.adagrad_acc ||
          d0.table_dtype != d.table_dtype || (d.table_dtype == EMB_DT_I8 && d0.row_scale != d.row_scale)) {
        free_plan(p);
        return EMB_ERR_INVALID_ARG;
      }
      p->col_table.push_back(it->second);
    }
  }
  if (base >= 0xFFFFFFFFull) {
    free_plan(p);
    return EMB_ERR_UNSUPPORTED;
  }
  p->n_tables = (int32_t)p->tables_h.size();
  p->table_base_h.push_back((uint32_t)base);
  p->key_total = (uint32_t)base;
  p->key_bits = 1;
  while (p->key_bits < 32 && (uint64_t(1) << p->key_bits) <= base) ++p->key_bits;

  // Column metadata, stream membership and output layout.
  std::vector<int32_t> stream_cols[2];
  int64_t out_col = 0, seq_unit = 0;
  p->meta_h.resize(n_cols);
  for (int32_t c = 0; c < n_cols; ++c) {
    const emb_column_desc& d = cols[c];
    ColMeta& m = p->meta_h[c];
    m.weight = d.weight;
    m.acc = d.adagrad_acc;
    m.qscale = d.table_dtype == EMB_DT_I8 ? d.row_scale : nullptr;
    m.dtype = d.table_dtype;
    if (d.table_dtype != EMB_DT_F32) p->low_precision = true;
    m.dflt = d.default_vec;
    m.bnd = d.boundaries;
    m.num_rows = d.num_rows;
    m.mod = make_div_magic((uint64_t)d.num_rows);
    m.dim = d.dim;
    m.dim4 = d.dim / 4;
    m.nb = d.transform == EMB_T_BUCKETIZE ? d.num_boundaries : 0;
    m.transform = d.transform;
    m.pooling = d.pooling;
    m.pad_len = d.pooling == EMB_POOL_NONE_PADDED ? d.pad_len : 0;
    m.trunc = d.pooling == EMB_POOL_NONE_PADDED ? 0 : d.max_len;
    m.table = p->col_table[c];
    m.table_base = p->table_base_h[m.table];
    m.col = c;
    if (d.pooling == EMB_POOL_NONE_PADDED) {
      m.out_col = -1;
      m.seq_unit = seq_unit;
      seq_unit += (int64_t)d.pad_len * d.dim;
      p->n_padded++;
    } else {
      m.out_col = (int32_t)out_col;
      m.seq_unit = 0;
      out_col += d.dim;
    }
    p->max_dim = std::max(p->max_dim, d.dim);
    stream_cols[d.transform == EMB_T_BUCKETIZE ? 1 : 0].push_back(c);
  }
  p->out_width = out_col;
  p->seq_per_bag = seq_unit;
  if (out_col >= (int64_t(1) << 31)) {
    free_plan(p);
    return EMB_ERR_UNSUPPORTED;
  }
  p->n_stream_cols[0] = (int32_t)stream_cols[0].size();
  p->n_stream_cols[1] = (int32_t)stream_cols[1].size();
  std::vector<int32_t> sc(stream_cols[0]);
  sc.insert(sc.end(), stream_cols[1].begin(), stream_cols[1].end());

  size_t total = 0;
  cudaError_t e = cudaSuccess;
  int dev = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = dmalloc(&p->meta_d, n_cols, &total);
  if (e == cudaSuccess) e = dmalloc(&p->colg_d, n_cols, &total);
  if (e == cudaSuccess) e = dmalloc(&p->tables_d, p->tables_h.size(), &total);
  if (e == cudaSuccess) e = dmalloc(&p->table_base_d, p->table_base_h.size(), &total);
  if (e == cudaSuccess) e = dmalloc(&p->status_d, 1, &total);
  if (e == cudaSuccess) e = dmalloc(&p->fwd_ticket, 2, &total);
  if (e == cudaSuccess) e = cudaMemset(p->fwd_ticket, 0, 2 * sizeof(unsigned long long));
  if (e == cudaSuccess) {
    // the forward reads a column's metadata by its position in its stream
    std::vector<ColMeta> ms(sc.size());
    for (size_t i = 0; i < sc.size(); ++i) ms[i] = p->meta_h[sc[i]];
    e = cudaMemcpy(p->meta_d, ms.data(), sizeof(ColMeta) * ms.size(), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess && !sc.empty()) {
    // work order of the forward's bag tiles: within each stream, the columns
    // with the widest stored rows first (ties in plan order)
    std::vector<int32_t> order;
    for (int st = 0; st < 2; ++st) {
      std::vector<int32_t> pos(stream_cols[st].size());
      for (size_t i = 0; i < pos.size(); ++i) pos[i] = (int32_t)i;
      auto row_bytes = [&](int32_t i) {
        const emb_column_desc& d = cols[stream_cols[st][i]];
        const int64_t el = d.table_dtype == EMB_DT_F32 ? 4 : d.table_dtype == EMB_DT_I8 ? 1 : 2;
        return (int64_t)d.dim * el;
      };
      std::stable_sort(pos.begin(), pos.end(), [&](int32_t x, int32_t y) { return row_bytes(x) > row_bytes(y); });
      order.insert(order.end(), pos.begin(), pos.end());
    }
    e = dmalloc(&p->col_order_d, order.size(), &total);
    if (e == cudaSuccess) e = cudaMemcpy(p->col_order_d, order.data(), sizeof(int32_t) * order.size(), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) {
    // long padded columns, by their position in meta_d
    std::vector<int32_t> pads;
    for (size_t i = 0; i < sc.size(); ++i) {
      const ColMeta& m = p->meta_h[sc[i]];
      if (m.pooling == EMB_POOL_NONE_PADDED && m.pad_len > kLongBag) {
        pads.push_back((int32_t)i);
        p->max_long_pad = std::max(p->max_long_pad, m.pad_len);
      }
    }
    p->n_long_padded = (int32_t)pads.size();
    for (int st = 0; st < 2; ++st) {
      bool all = !stream_cols[st].empty();
      for (int32_t c : stream_cols[st]) {
        const ColMeta& m = p->meta_h[c];
        all = all && m.pooling == EMB_POOL_NONE_PADDED && m.pad_len > kLongBag;
      }
      p->long_padded_only[st] = all;
    }
    if (!pads.empty()) {
      e = dmalloc(&p->pad_cols_d, pads.size(), &total);
      if (e == cudaSuccess)
        e = cudaMemcpy(p->pad_cols_d, pads.data(), sizeof(int32_t) * pads.size(), cudaMemcpyHostToDevice);
    }
  }
  if (e == cudaSuccess)
    e = cudaMemcpy(p->tables_d, p->tables_h.data(), sizeof(TableMeta) * p->tables_h.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(p->table_base_d, p->table_base_h.data(), sizeof(uint32_t) * p->table_base_h.size(),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(p->status_d, 0, sizeof(uint32_t));
  if (e == cudaSuccess) {
    std::vector<int4> cg(n_cols);
    for (int32_t c = 0; c < n_cols; ++c)
      cg[c] = make_int4(p->meta_h[c].out_col, cols[c].pooling == EMB_POOL_MEAN ? 1 : 0, cols[c].dim / 4, 0);
    e = cudaMemcpy(p->colg_d, cg.data(), sizeof(int4) * n_cols, cudaMemcpyHostToDevice);
  }

  if (e == cudaSuccess && training) {
    Workspace& w = p->ws;
    const int64_t n = std::max<int64_t>(max_ids, 1);
    w.max_tiles = (n + kSortTile - 1) / kSortTile;
    w.n_units_max = (n + kUnit - 1) / kUnit;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
      e = dmalloc(&w.keys[i], n, &total);
      if (e == cudaSuccess) e = dmalloc(&w.vals[i], n, &total);
    }
    if (e == cudaSuccess) e = dmalloc(&w.inv_n, (size_t)n_cols * max_batch, &total);
    if (e == cudaSuccess) e = dmalloc(&w.rec_src, n, &total);
    if (e == cudaSuccess) e = dmalloc(&w.hist, sort_scratch_words<uint32_t>(p->key_bits, n), &total);
    if (e == cudaSuccess) e = dmalloc(&w.run_head, n + 1, &total);
    if (e == cudaSuccess) e = dmalloc(&w.head_pos, n, &total);
    if (e == cudaSuccess) e = dmalloc(&w.n_runs, 4, &total);
    if (e == cudaSuccess) e = dmalloc(&w.scan_part, (n + 1023) / 1024 + 64, &total);
    if (e == cudaSuccess) e = dmalloc(&w.partial, (size_t)w.n_units_max * 2 * (p->max_dim / 4), &total);
    if (e == cudaSuccess) e = dmalloc(&w.part_pos, (size_t)w.n_units_max * 2, &total);
    if (e == cudaSuccess) e = dmalloc(&w.part_thru, (size_t)w.n_units_max, &total);
    if (e == cudaSuccess && (flags & EMB_PLAN_ATOMIC_BACKWARD)) {
      p->atomic_bwd = true;
      const size_t words = ((size_t)p->key_total + 31) / 32;
      const size_t cg = (size_t)n * p->max_dim;
      e = dmalloc(&w.touched, words, &total);
      if (e == cudaSuccess) e = cudaMemset(w.touched, 0, sizeof(uint32_t) * std::max<size_t>(words, 1));
      if (e == cudaSuccess) e = dmalloc(&w.bit_part, (words + 1023) / 1024, &total);
      if (e == cudaSuccess) e = dmalloc(&w.n_uniq, 1, &total);
      if (e == cudaSuccess) e = dmalloc(&w.uniq, n, &total);
      if (e == cudaSuccess) e = dmalloc(&w.slot_of, (size_t)p->key_total, &total);
      if (e == cudaSuccess) e = dmalloc(&w.cgrad, cg, &total);
      if (e == cudaSuccess) e = cudaMemset(w.cgrad, 0, sizeof(float) * std::max<size_t>(cg, 1));
      if (e == cudaSuccess) e = dmalloc(&w.ucount, n, &total);
      if (e == cudaSuccess) e = cudaMemset(w.ucount, 0, sizeof(uint32_t) * n);
    }
  }
  p->ws.bytes = total;
  if (e == cudaSuccess) p->fwd_ctas_per_sm = forward_ctas_per_sm();
  if (e != cudaSuccess) {
    free_plan(p);
    cudaGetLastError();
    return cuda_status(e);
  }
  *out = p;
  return EMB_OK;
}

extern "C" emb_status emb_plan_destroy(emb_plan p) {
  if (!p) return EMB_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  free_plan(p);
  return EMB_OK;
}

extern "C" emb_status emb_plan_info(emb_plan p, int64_t* out_width, int64_t* seq_floats_per_bag,
                                    int32_t* n_tables, int32_t* col_table, int64_t* workspace_bytes) {
  if (!p) return EMB_ERR_INVALID_ARG;
  if (out_width) *out_width = p->out_width;
  if (seq_floats_per_bag) *seq_floats_per_bag = p->seq_per_bag;
  if (n_tables) *n_tables = p->n_tables;
  if (col_table) std::memcpy(col_table, p->col_table.data(), sizeof(int32_t) * p->n_cols);
  if (workspace_bytes) *workspace_bytes = (int64_t)p->ws.bytes;
  return EMB_OK;
}

extern "C" emb_status emb_forward(emb_plan p, int32_t batch, const int64_t* ids,
                                  const int32_t* id_offsets, const float* id_weights, int64_t n_ids,
                                  const float* fvals, const int32_t* f_offsets, const float* f_weights,
                                  int64_t n_fvals, float* out, float* seq_out, int64_t* rows_dbg,
                                  void* stream) {
  if (!p || batch < 0 || batch > p->max_batch || n_ids < 0 || n_fvals < 0) return EMB_ERR_INVALID_ARG;
  if (n_ids >= (int64_t(1) << 31) || n_fvals >= (int64_t(1) << 31)) return EMB_ERR_UNSUPPORTED;
  if (p->n_stream_cols[0] > 0 && (!id_offsets || (n_ids > 0 && !ids))) return EMB_ERR_INVALID_ARG;
  if (p->n_stream_cols[1] > 0 && (!f_offsets || (n_fvals > 0 && !fvals))) return EMB_ERR_INVALID_ARG;
  if (p->out_width > 0 && batch > 0 && (!out || !aligned16(out))) return EMB_ERR_INVALID_ARG;
  if (p->n_padded > 0 && batch > 0 && (!seq_out || !aligned16(seq_out))) return EMB_ERR_INVALID_ARG;
  if (p->training) {
    if (n_ids + n_fvals > p->max_ids) return EMB_ERR_INVALID_ARG;
    // padded gradient sources are addressed in float4 units below 2^31
    if (p->seq_per_bag * (int64_t)batch / 4 >= (int64_t(1) << 31)) return EMB_ERR_UNSUPPORTED;
  }
  if (n_ids == 0) id_weights = nullptr;
  if (n_fvals == 0) f_weights = nullptr;
  emb_status s = launch_forward(p, batch, ids, id_offsets, id_weights, n_ids, fvals, f_offsets, f_weights,
                                n_fvals, out, seq_out, rows_dbg, (cudaStream_t)stream);
  if (s == EMB_OK && p->training) {
    p->have_forward = true;
    p->last_batch = batch;
    p->last_n = n_ids + n_fvals;
    p->last_n_ids = n_ids;
    p->last_weighted = id_weights || f_weights;
  }
  return s;
}

extern "C" emb_status emb_backward_update(emb_plan p, const float* grad_out, const float* grad_seq,
                                          float lr, float eps, void* stream,
                                          const emb_backward_debug* dbg) {
  if (!p || !p->training || !p->have_forward) return EMB_ERR_INVALID_ARG;
  if (p->last_batch > 0 && p->out_width > 0 && !grad_out) return EMB_ERR_INVALID_ARG;
  if (p->last_batch > 0 && p->n_padded > 0 && !grad_seq) return EMB_ERR_INVALID_ARG;
  if (!(lr == lr) || !(eps == eps)) return EMB_ERR_INVALID_ARG;
  if (p->atomic_bwd) return launch_backward_atomic(p, grad_out, grad_seq, lr, eps, (cudaStream_t)stream, dbg);
  return launch_backward(p, grad_out, grad_seq, lr, eps, (cudaStream_t)stream, dbg);
}

extern "C" emb_status emb_get_device_status(emb_plan p, void* stream) {
  if (!p) return EMB_ERR_INVALID_ARG;
  uint32_t st = 0;
  EMB_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
  EMB_CUDA_TRY(cudaMemcpy(&st, p->status_d, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  EMB_CUDA_TRY(cudaMemset(p->status_d, 0, sizeof(uint32_t)));
  return (emb_status)st;
}

extern "C" emb_status emb_selftest_hash_mod(const int64_t* ids, int64_t n, int64_t num_rows,
                                            int64_t* rows_out) {
  if (n < 0 || num_rows < 1 || (n > 0 && (!ids || !rows_out))) return EMB_ERR_INVALID_ARG;
  DivMagic g = make_div_magic((uint64_t)num_rows);
  for (int64_t i = 0; i < n; ++i) rows_out[i] = (int64_t)mod_magic(splitmix64((uint64_t)ids[i]), g);
  return EMB_OK;
}

extern "C" const char* emb_version(void) { return "sparse_lookup_gb300 0.1 (sm_103a)"; }
