// hash.cu -- K-H: the collision-free dynamic table (Monolith §2.1 "Tabel Hash").
#include "common.cuh"

extern "C" emb_status hash_create(int64_t, int64_t, int32_t, int32_t, int32_t, uint64_t, float, emb_hash* out) {
  if (out) *out = nullptr;
  return EMB_ERR_UNSUPPORTED;
}
extern "C" emb_status hash_rows(emb_hash, float**, float**) { return EMB_ERR_UNSUPPORTED; }
extern "C" emb_status hash_lookup_or_insert(emb_hash, const int32_t*, const int64_t*, int64_t, uint32_t,
                                            int64_t*, void*) { return EMB_ERR_UNSUPPORTED; }
extern "C" emb_status hash_evict_expired(emb_hash, uint32_t, uint32_t, void*, int64_t*) { return EMB_ERR_UNSUPPORTED; }
extern "C" emb_status hash_export(emb_hash, int32_t*, int64_t*, int64_t*, int32_t*, uint32_t*, int64_t, int64_t*,
                                  void*) { return EMB_ERR_UNSUPPORTED; }
extern "C" emb_status hash_get_device_status(emb_hash, void*) { return EMB_ERR_UNSUPPORTED; }
extern "C" emb_status hash_destroy(emb_hash) { return EMB_ERR_UNSUPPORTED; }
