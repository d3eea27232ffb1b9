// C ABI of libvitfe: handle lifetime, argument validation, launches.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "vitfe_internal.cuh"

struct vitfe_ctx {
  vitfe::Ctx c;
};

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kMaxRows = 0x7fffffffLL - 1024;

void free_ctx(vitfe_ctx* h) {
  if (!h) return;
  if (h->c.w_tile) cudaFree(h->c.w_tile);
  if (h->c.w_tile_f) cudaFree(h->c.w_tile_f);
  if (h->c.bias) cudaFree(h->c.bias);
  if (h->c.rope_tab) cudaFree(h->c.rope_tab);
  delete h;
}

vitfe_status check_common(vitfe_t h, const vitfe_item* items, const int32_t* n_items, int32_t max_items,
                          int64_t rows) {
  if (h == nullptr || items == nullptr || n_items == nullptr) return VITFE_EINVAL;
  if (max_items < 0 || max_items > VITFE_MAX_ITEMS) return VITFE_EINVAL;
  if (rows < 0 || rows > kMaxRows) return VITFE_EINVAL;
  if (!aligned(items, 8) || !aligned(n_items, 4)) return VITFE_EINVAL;
  return VITFE_OK;
}

vitfe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? VITFE_OK : VITFE_ECUDA; }

}  // namespace

extern "C" {

const char* vitfe_status_str(vitfe_status s) {
  switch (s) {
    case VITFE_OK: return "ok";
    case VITFE_EINVAL: return "invalid argument";
    case VITFE_ENOMEM: return "device allocation failed";
    case VITFE_ECUDA: return "CUDA runtime error";
    case VITFE_EDEVICE_DESC: return "inconsistent item descriptor (device)";
    case VITFE_EDEVICE_RANGE: return "pixels or rows out of range (device)";
    case VITFE_EDEVICE_TIMEOUT: return "pipeline wait timed out (device)";
    case VITFE_EUNSUPPORTED: return "unsupported shape";
  }
  return "unknown status";
}

int vitfe_feature_dim(vitfe_t h) { return h ? h->c.K : 0; }

vitfe_status vitfe_create(vitfe_t* out, const float mean[3], const float std_[3], float rescale, int patch,
                          int tpatch, int merge, int hidden, const void* W, const void* b, cudaStream_t stream) {
  if (out == nullptr) return VITFE_EINVAL;
  *out = nullptr;
  if (mean == nullptr || std_ == nullptr || W == nullptr) return VITFE_EINVAL;
  for (int c = 0; c < 3; ++c) {
    if (!std::isfinite(mean[c]) || !std::isfinite(std_[c]) || !(std_[c] > 0.0f)) return VITFE_EINVAL;
  }
  if (!std::isfinite(rescale) || !(rescale > 0.0f)) return VITFE_EINVAL;
  if (patch < 1 || patch > 32 || tpatch < 1 || tpatch > 4 || merge < 1 || merge > 8) return VITFE_EINVAL;
  if (hidden < 16 || hidden > 8192 || (hidden % 16) != 0) return VITFE_EINVAL;
  if (!aligned(W, 2) || (b && !aligned(b, 2))) return VITFE_EINVAL;

  vitfe_ctx* h = new (std::nothrow) vitfe_ctx();
  if (!h) return VITFE_ENOMEM;
  vitfe::Ctx& c = h->c;
  if (cudaGetDevice(&c.device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c.sm_count, cudaDevAttrMultiProcessorCount, c.device) != cudaSuccess) {
    free_ctx(h);
    return VITFE_ECUDA;
  }
  for (int ch = 0; ch < 3; ++ch) {
    c.scale[ch] = (float)((double)rescale / (double)std_[ch]);
    c.shift[ch] = (float)(-(double)mean[ch] / (double)std_[ch]);
  }
  c.P = patch;
  c.T = tpatch;
  c.M = merge;
  c.N = hidden;
  c.kslice = 3 * patch * patch;
  c.kslice_pad = (c.kslice + 63) / 64 * 64;
  c.nblk = c.kslice_pad / 64;
  c.K = tpatch * c.kslice;
  if (const char* env = std::getenv("VITFE_WAIT_LIMIT_MS")) {
    const long ms = std::strtol(env, nullptr, 10);
    if (ms > 0) c.wait_limit_ns = (uint64_t)ms * 1000000ull;
  }

  if (cudaMalloc(&c.bias, (size_t)c.N * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&c.rope_tab, (size_t)(vitfe::Ctx::kRopeSlots + 1) * 2 * VITFE_ROPE_MAX_SIDE * (VITFE_ROPE_MAX_HEAD_DIM / 4) *
                                  sizeof(float)) !=
          cudaSuccess) {
    cudaGetLastError();
    free_ctx(h);
    return VITFE_ENOMEM;
  }
  // the embed kernel's tile shape decides the weight layout
  cudaError_t e = vitfe::embed_configure(c);
  if (e != cudaSuccess) {
    free_ctx(h);
    return VITFE_ECUDA;
  }
  if (c.embed_ok) {
    const size_t npass = (size_t)((c.N + c.bn - 1) / c.bn);
    c.w_tile_bytes = npass * 2 * (size_t)c.T * (size_t)c.nblk * (size_t)(c.bn / 2) * 128;
    c.w_tile_f_bytes = c.T > 1 ? c.w_tile_bytes / (size_t)c.T : 0;
    if (cudaMalloc(&c.w_tile, c.w_tile_bytes) != cudaSuccess ||
        (c.w_tile_f_bytes > 0 && cudaMalloc(&c.w_tile_f, c.w_tile_f_bytes) != cudaSuccess)) {
      cudaGetLastError();
      free_ctx(h);
      return VITFE_ENOMEM;
    }
    e = vitfe::launch_tile_weight(c, static_cast<const __nv_bfloat16*>(W), static_cast<const __nv_bfloat16*>(b),
                                  stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
      free_ctx(h);
      return VITFE_ECUDA;
    }
    EncodeTiledFn enc = get_encode_tiled();
    if (enc == nullptr) {
      free_ctx(h);
      return VITFE_ECUDA;
    }
    // the tiled weight as rows of 512 bytes: one box (bn/8 rows) is one shared-memory image
    const cuuint64_t rows512 = (cuuint64_t)(c.w_tile_bytes / 512);
    const cuuint64_t gdim[2] = {256u, rows512};
    const cuuint64_t gstride[1] = {512u};
    const cuuint32_t box[2] = {256u, (cuuint32_t)(c.bn / 8)};
    const cuuint32_t estride[2] = {1u, 1u};
    CUresult r = enc(&c.tmap_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.w_tile, gdim, gstride, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS && c.w_tile_f != nullptr) {
      const cuuint64_t gdim_f[2] = {256u, (cuuint64_t)(c.w_tile_f_bytes / 512)};
      r = enc(&c.tmap_wf, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.w_tile_f, gdim_f, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) {
      free_ctx(h);
      return VITFE_ECUDA;
    }
  }
  *out = h;
  return VITFE_OK;
}

void vitfe_destroy(vitfe_t h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_ctx(h);
}

vitfe_status vitfe_embed(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes, const vitfe_item* items,
                         const int32_t* n_items, int32_t max_items, int64_t rows, void* out, int32_t* status,
                         cudaStream_t stream) {
  vitfe_status st = check_common(h, items, n_items, max_items, rows);
  if (st != VITFE_OK) return st;
  if (pixels == nullptr || pixel_bytes < 0 || !aligned(pixels, 16)) return VITFE_EINVAL;
  if ((out == nullptr && rows > 0) || !aligned(out, 16)) return VITFE_EINVAL;
  if (status && !aligned(status, 4)) return VITFE_EINVAL;
  if (!h->c.embed_ok) return VITFE_EUNSUPPORTED;
  return from_cuda(vitfe::launch_embed(h->c, pixels, pixel_bytes, items, n_items, max_items, rows, out, status,
                                       stream));
}

vitfe_status vitfe_embed_folded(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes, const vitfe_item* items,
                                const int32_t* n_items, int32_t max_items, int64_t rows, void* out,
                                int32_t* status, cudaStream_t stream) {
  vitfe_status st = check_common(h, items, n_items, max_items, rows);
  if (st != VITFE_OK) return st;
  if (pixels == nullptr || pixel_bytes < 0 || !aligned(pixels, 16)) return VITFE_EINVAL;
  if ((out == nullptr && rows > 0) || !aligned(out, 16)) return VITFE_EINVAL;
  if (status && !aligned(status, 4)) return VITFE_EINVAL;
  if (!h->c.embed_ok || h->c.w_tile_f == nullptr) return VITFE_EUNSUPPORTED;
  return from_cuda(vitfe::launch_embed(h->c, pixels, pixel_bytes, items, n_items, max_items, rows, out, status,
                                       stream, nullptr, 0, nullptr, nullptr, true));
}

vitfe_status vitfe_embed_rope(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes, const vitfe_item* items,
                              const int32_t* n_items, int32_t max_items, int64_t rows, void* out, int head_dim,
                              float theta, float* cos, float* sin, int32_t* status, cudaStream_t stream) {
  vitfe_status st = check_common(h, items, n_items, max_items, rows);
  if (st != VITFE_OK) return st;
  if (pixels == nullptr || pixel_bytes < 0 || !aligned(pixels, 16)) return VITFE_EINVAL;
  if ((out == nullptr && rows > 0) || !aligned(out, 16)) return VITFE_EINVAL;
  if (head_dim < 8 || head_dim > VITFE_ROPE_MAX_HEAD_DIM || (head_dim % 8) != 0) return VITFE_EINVAL;
  if (!std::isfinite(theta) || !(theta > 0.0f)) return VITFE_EINVAL;
  if (rows > 0 && (cos == nullptr || sin == nullptr)) return VITFE_EINVAL;
  if (!aligned(cos, 16) || !aligned(sin, 16)) return VITFE_EINVAL;
  if (status && !aligned(status, 4)) return VITFE_EINVAL;
  if (!h->c.embed_ok) return VITFE_EUNSUPPORTED;
  const float* tab = nullptr;
  cudaError_t e = vitfe::rope_table_for(h->c, head_dim, theta, stream, &tab);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(vitfe::launch_embed(h->c, pixels, pixel_bytes, items, n_items, max_items, rows, out, status,
                                       stream, tab, head_dim / 4, cos, sin));
}

vitfe_status vitfe_rope(vitfe_t h, const vitfe_item* items, const int32_t* n_items, int32_t max_items,
                        int64_t rows, int head_dim, float theta, float* cos, float* sin, int32_t* status,
                        cudaStream_t stream) {
  vitfe_status st = check_common(h, items, n_items, max_items, rows);
  if (st != VITFE_OK) return st;
  if (head_dim < 8 || head_dim > VITFE_ROPE_MAX_HEAD_DIM || (head_dim % 8) != 0) return VITFE_EINVAL;
  if (!std::isfinite(theta) || !(theta > 0.0f)) return VITFE_EINVAL;
  if (rows > 0 && (cos == nullptr || sin == nullptr)) return VITFE_EINVAL;
  if (!aligned(cos, 16) || !aligned(sin, 16)) return VITFE_EINVAL;
  if (status && !aligned(status, 4)) return VITFE_EINVAL;
  return from_cuda(vitfe::launch_rope(h->c, items, n_items, max_items, rows, head_dim, theta, cos, sin, status,
                                      stream));
}

vitfe_status vitfe_normalize_patchify(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes,
                                      const vitfe_item* items, const int32_t* n_items, int32_t max_items,
                                      int64_t rows, void* out, int32_t* status, cudaStream_t stream) {
  vitfe_status st = check_common(h, items, n_items, max_items, rows);
  if (st != VITFE_OK) return st;
  if (pixels == nullptr || pixel_bytes < 0 || !aligned(pixels, 16)) return VITFE_EINVAL;
  if ((out == nullptr && rows > 0) || !aligned(out, 16)) return VITFE_EINVAL;
  if (status && !aligned(status, 4)) return VITFE_EINVAL;
  return from_cuda(vitfe::launch_normalize_patchify(h->c, pixels, pixel_bytes, items, n_items, max_items, rows,
                                                    out, status, stream));
}

vitfe_status vitfe_pos_ids(vitfe_t h, const vitfe_item* items, const int32_t* n_items, int32_t max_items,
                           int64_t rows, int32_t* pos, int32_t* status, cudaStream_t stream) {
  vitfe_status st = check_common(h, items, n_items, max_items, rows);
  if (st != VITFE_OK) return st;
  if ((pos == nullptr && rows > 0) || !aligned(pos, 8)) return VITFE_EINVAL;
  if (status && !aligned(status, 4)) return VITFE_EINVAL;
  return from_cuda(vitfe::launch_pos_ids(h->c, items, n_items, max_items, rows, pos, status, stream));
}

vitfe_status vitfe_cu_seqlens(vitfe_t h, const vitfe_item* items, const int32_t* n_items, int32_t max_items,
                              int64_t rows, int32_t max_seqs, int32_t* cu_seqlens, int32_t* seq_info,
                              int32_t* status, cudaStream_t stream) {
  vitfe_status st = check_common(h, items, n_items, max_items, rows);
  if (st != VITFE_OK) return st;
  if (max_seqs < 0 || max_seqs > kMaxRows) return VITFE_EINVAL;
  if (cu_seqlens == nullptr || seq_info == nullptr || !aligned(cu_seqlens, 4) || !aligned(seq_info, 4))
    return VITFE_EINVAL;
  if (status && !aligned(status, 4)) return VITFE_EINVAL;
  return from_cuda(vitfe::launch_cu_seqlens(h->c, items, n_items, max_items, rows, max_seqs, cu_seqlens, seq_info,
                                            status, stream));
}

vitfe_status vitfe_rope_apply(const float* cos, const float* sin, int64_t rows, int head_dim, void* q,
                              int32_t heads_q, int64_t q_row_stride, void* k, int32_t heads_k,
                              int64_t k_row_stride, cudaStream_t stream) {
  if (rows < 0 || rows > kMaxRows) return VITFE_EINVAL;
  if (head_dim < 8 || head_dim > VITFE_ROPE_MAX_HEAD_DIM || (head_dim % 8) != 0) return VITFE_EINVAL;
  if (heads_q < 0 || heads_k < 0 || heads_q > 4096 || heads_k > 4096) return VITFE_EINVAL;
  if (rows > 0 && (cos == nullptr || sin == nullptr)) return VITFE_EINVAL;
  if (!aligned(cos, 16) || !aligned(sin, 16)) return VITFE_EINVAL;
  if (heads_q > 0) {
    if (q == nullptr || !aligned(q, 8) || q_row_stride < (int64_t)heads_q * head_dim || (q_row_stride % 4) != 0)
      return VITFE_EINVAL;
  }
  if (heads_k > 0) {
    if (k == nullptr || !aligned(k, 8) || k_row_stride < (int64_t)heads_k * head_dim || (k_row_stride % 4) != 0)
      return VITFE_EINVAL;
  }
  return from_cuda(vitfe::launch_rope_apply(cos, sin, rows, head_dim, q, heads_q, q_row_stride, k, heads_k,
                                            k_row_stride, stream));
}

vitfe_status vitfe_items_from_grid(const int32_t* grid_thw, const uint8_t* is_still, int32_t n, int patch,
                                   int tpatch, vitfe_item* items_out, int64_t* total_rows, int64_t* pixel_bytes) {
  if (n < 0 || (n > 0 && (grid_thw == nullptr || items_out == nullptr)) || total_rows == nullptr ||
      pixel_bytes == nullptr || patch < 1 || tpatch < 1)
    return VITFE_EINVAL;
  int64_t off = 0, rows = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t t = grid_thw[3 * i], hh = grid_thw[3 * i + 1], ww = grid_thw[3 * i + 2];
    if (t < 0 || hh < 0 || ww < 0) return VITFE_EINVAL;
    const bool still = is_still ? (is_still[i] != 0) : (t == 1);
    if (still && t != 1) return VITFE_EINVAL;
    const int64_t frames = still ? 1 : t * tpatch;
    if (frames > 0x7fffffffLL) return VITFE_EINVAL;
    items_out[i].pixel_offset = off;
    items_out[i].t = (int32_t)t;
    items_out[i].h = (int32_t)hh;
    items_out[i].w = (int32_t)ww;
    items_out[i].frames = (int32_t)frames;
    off += (frames * (hh * patch) * (ww * patch) * 3 + 15) / 16 * 16;
    rows += t * hh * ww;
  }
  *total_rows = rows;
  *pixel_bytes = off;
  return VITFE_OK;
}

}  // extern "C"
