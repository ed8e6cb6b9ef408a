// Host-side checks shared by every entry point, status strings, version.
#include "se_common.cuh"

se_status se_check_kv(const se_paged_kv* kv) {
  if (kv == nullptr) return SE_ERR_INVALID_ARG;
  if (kv->k_pool == nullptr || kv->v_pool == nullptr || kv->block_table == nullptr ||
      kv->slot_map == nullptr || kv->ctx_len == nullptr || kv->logical_len == nullptr ||
      kv->free_list == nullptr || kv->free_top == nullptr || kv->status == nullptr)
    return SE_ERR_INVALID_ARG;
  if (kv->B < 1 || kv->Hkv < 1 || kv->Hq < kv->Hkv || kv->Hq % kv->Hkv != 0 ||
      kv->num_pages < 1 || kv->max_pages_per_seq < 1)
    return SE_ERR_INVALID_ARG;
  if (kv->dtype != SE_BF16 && kv->dtype != SE_F32) return SE_ERR_UNSUPPORTED;
  if (kv->D != 64 && kv->D != 128) return SE_ERR_UNSUPPORTED;
  const int P = kv->page_size;
  if (P < 1 || P > 64 || (P & (P - 1)) != 0) return SE_ERR_UNSUPPORTED;
  if ((int64_t)kv->max_pages_per_seq * P > (int64_t)1 << 30) return SE_ERR_UNSUPPORTED;
  return SE_OK;
}

se_status se_last_launch_status() {
  return cudaGetLastError() == cudaSuccess ? SE_OK : SE_ERR_CUDA;
}

extern "C" const char* se_status_string(int32_t status) {
  switch (status) {
    case SE_OK: return "SE_OK";
    case SE_ERR_INVALID_ARG: return "SE_ERR_INVALID_ARG";
    case SE_ERR_UNSUPPORTED: return "SE_ERR_UNSUPPORTED";
    case SE_ERR_OUT_OF_PAGES: return "SE_ERR_OUT_OF_PAGES";
    case SE_ERR_UNEVEN: return "SE_ERR_UNEVEN";
    case SE_ERR_BUSY: return "SE_ERR_BUSY";
    case SE_ERR_TIMEOUT: return "SE_ERR_TIMEOUT";
    case SE_ERR_BOUNDS: return "SE_ERR_BOUNDS";
    case SE_ERR_CUDA: return "SE_ERR_CUDA";
    default: return "SE_ERR_UNKNOWN";
  }
}

extern "C" int32_t se_version(void) { return 100; }
