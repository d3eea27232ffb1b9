// C ABI of libvitfe: handle lifetime, argument validation, launches.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

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

void free_pipe_buffers(vitfe::Ctx::HostPipe& p) {
  for (int b = 0; b < 2; ++b) {
    if (p.px[b]) cudaFree(p.px[b]);
    if (p.out[b]) cudaFree(p.out[b]);
    if (p.cos[b]) cudaFree(p.cos[b]);
    if (p.sin[b]) cudaFree(p.sin[b]);
    p.px[b] = nullptr;
    p.out[b] = nullptr;
    p.cos[b] = p.sin[b] = nullptr;
  }
  p.px_cap = 0;
  p.rows_cap = 0;
  p.hd_cap = 0;
}

void free_pipe(vitfe::Ctx::HostPipe& p) {
  free_pipe_buffers(p);
  for (int b = 0; b < 2; ++b) {
    if (p.items[b]) cudaFree(p.items[b]);
    if (p.n[b]) cudaFree(p.n[b]);
    if (p.status[b]) cudaFree(p.status[b]);
    if (p.up[b]) cudaEventDestroy(p.up[b]);
    if (p.done[b]) cudaEventDestroy(p.done[b]);
    if (p.down[b]) cudaEventDestroy(p.down[b]);
  }
  if (p.h_items) cudaFreeHost(p.h_items);
  if (p.h_small) cudaFreeHost(p.h_small);
  if (p.h2d) cudaStreamDestroy(p.h2d);
  if (p.comp) cudaStreamDestroy(p.comp);
  if (p.d2h) cudaStreamDestroy(p.d2h);
  p = vitfe::Ctx::HostPipe();
}

void free_ctx(vitfe_ctx* h) {
  if (!h) return;
  free_pipe(h->c.pipe);
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

namespace {

vitfe_status pipe_ready(vitfe::Ctx& c, size_t px_bytes, int64_t rows, int head_dim) {
  auto& p = c.pipe;
  if (!p.ready) {
    bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess;
    for (int b = 0; ok && b < 2; ++b)
      ok = cudaEventCreateWithFlags(&p.up[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.done[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.down[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaMalloc(&p.items[b], sizeof(vitfe_item) * VITFE_MAX_ITEMS) == cudaSuccess &&
           cudaMalloc(&p.n[b], sizeof(int32_t)) == cudaSuccess &&
           cudaMalloc(&p.status[b], 2 * sizeof(int32_t)) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      free_pipe(p);
      return VITFE_ENOMEM;
    }
    p.ready = true;
  }
  if (px_bytes > p.px_cap || rows > p.rows_cap || head_dim > p.hd_cap) {
    // grow: nothing of this handle's pipeline may still be in flight
    if (cudaStreamSynchronize(p.h2d) != cudaSuccess || cudaStreamSynchronize(p.comp) != cudaSuccess ||
        cudaStreamSynchronize(p.d2h) != cudaSuccess)
      return VITFE_ECUDA;
    const size_t pxc = px_bytes > p.px_cap ? px_bytes : p.px_cap;
    const int64_t rc = rows > p.rows_cap ? rows : p.rows_cap;
    const int hc = head_dim > p.hd_cap ? head_dim : p.hd_cap;
    free_pipe_buffers(p);
    bool ok = true;
    for (int b = 0; ok && b < 2; ++b)
      ok = cudaMalloc(&p.px[b], pxc > 16 ? pxc : 16) == cudaSuccess &&
           cudaMalloc(&p.out[b], (size_t)(rc > 1 ? rc : 1) * c.N * sizeof(__nv_bfloat16)) == cudaSuccess &&
           cudaMalloc(&p.cos[b], (size_t)(rc > 1 ? rc : 1) * (hc / 2) * sizeof(float)) == cudaSuccess &&
           cudaMalloc(&p.sin[b], (size_t)(rc > 1 ? rc : 1) * (hc / 2) * sizeof(float)) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      free_pipe_buffers(p);
      return VITFE_ENOMEM;
    }
    p.px_cap = pxc;
    p.rows_cap = rc;
    p.hd_cap = hc;
  }
  return VITFE_OK;
}

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
  if (const char* env = std::getenv("VITFE_TEST_STALL_W_LOADS")) c.test_stall_w_loads = env[0] == '1';

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
  if (e == cudaSuccess) e = vitfe::np_configure(c);
  if (e != cudaSuccess) {
    free_ctx(h);
    return VITFE_ECUDA;
  }
  if (c.embed_ok) {
    const size_t npass = (size_t)((c.N + c.bn - 1) / c.bn);
    const size_t img_bytes = (size_t)(c.bn / 2) * 128;
    c.w_tile_bytes = npass * 2 * (size_t)vitfe::w_images(c.kslice, c.T) * img_bytes;
    c.w_tile_f_bytes = c.T > 1 ? npass * 2 * (size_t)vitfe::w_images(c.kslice, 1) * img_bytes : 0;
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

// ---------------------------------------------------------------------------
// Host-buffer pipeline: the items are cut into `chunks` runs of consecutive items with
// about equal rows.  Chunk c uses device staging set c % 2: its pixels and descriptors go
// up on one stream, the fused embed + RoPE launch runs on a second, the results come down
// on a third, so chunk c's upload and launch overlap chunk c - 1's download.
// ---------------------------------------------------------------------------

vitfe_status vitfe_embed_rope_host(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes, const vitfe_item* items,
                                   int32_t n_items, void* out, int head_dim, float theta, float* cos, float* sin,
                                   int32_t* status, int32_t chunks) {
  if (h == nullptr || n_items < 0 || n_items > VITFE_MAX_HOST_ITEMS || (n_items > 0 && items == nullptr))
    return VITFE_EINVAL;
  if (pixel_bytes < 0 || (pixel_bytes > 0 && pixels == nullptr) || chunks < 1) return VITFE_EINVAL;
  if (head_dim < 8 || head_dim > VITFE_ROPE_MAX_HEAD_DIM || (head_dim % 8) != 0) return VITFE_EINVAL;
  if (!std::isfinite(theta) || !(theta > 0.0f)) return VITFE_EINVAL;
  vitfe::Ctx& c = h->c;
  if (!c.embed_ok) return VITFE_EUNSUPPORTED;
  // host-side validation: every item's pixels lie inside the host buffer
  std::vector<int64_t> row0((size_t)n_items + 1, 0), pend((size_t)n_items, 0);
  for (int i = 0; i < n_items; ++i) {
    const vitfe_item& it = items[i];
    if (it.t < 0 || it.h < 0 || it.w < 0 || it.frames < 1 || it.pixel_offset < 0 || (it.pixel_offset & 15))
      return VITFE_EINVAL;
    const int64_t r = (int64_t)it.t * it.h * it.w;
    const int64_t bytes = (int64_t)it.frames * it.h * c.P * it.w * c.P * 3;
    if (it.pixel_offset + bytes > pixel_bytes) return VITFE_EINVAL;
    row0[i + 1] = row0[i] + r;
    pend[i] = it.pixel_offset + bytes;
    if (row0[i + 1] > kMaxRows) return VITFE_EINVAL;
  }
  const int64_t rows = row0[n_items];
  if (rows > 0 && (out == nullptr || cos == nullptr || sin == nullptr)) return VITFE_EINVAL;
  if (status != nullptr) {
    status[0] = 0;
    status[1] = -1;
  }
  if (n_items == 0) return VITFE_OK;
  // chunk boundaries: runs of consecutive items with about rows / chunks rows, at most
  // VITFE_MAX_ITEMS items each
  std::vector<int> cut{0};
  for (int i = 1; i < n_items; ++i) {
    const int64_t target = rows * (int64_t)cut.size() / chunks;
    if (row0[i] >= target || i - cut.back() >= VITFE_MAX_ITEMS) cut.push_back(i);
  }
  cut.push_back(n_items);
  const int nch = (int)cut.size() - 1;
  size_t px_max = 0;
  int64_t rows_max = 0;
  std::vector<int64_t> base((size_t)nch), span((size_t)nch);
  for (int k = 0; k < nch; ++k) {
    int64_t lo = items[cut[k]].pixel_offset, hi = lo;
    for (int i = cut[k]; i < cut[k + 1]; ++i) {
      lo = items[i].pixel_offset < lo ? items[i].pixel_offset : lo;
      hi = pend[i] > hi ? pend[i] : hi;
    }
    base[k] = lo;
    span[k] = (hi - lo + 15) / 16 * 16;
    if (lo + span[k] > pixel_bytes) span[k] = pixel_bytes - lo;   // the last bytes of the buffer
    px_max = (size_t)span[k] > px_max ? (size_t)span[k] : px_max;
    const int64_t r = row0[cut[k + 1]] - row0[cut[k]];
    rows_max = r > rows_max ? r : rows_max;
  }
  vitfe_status st = pipe_ready(c, px_max, rows_max, head_dim);
  if (st != VITFE_OK) return st;
  auto& p = c.pipe;
  if ((size_t)n_items > p.h_items_cap) {
    if (p.h_items) cudaFreeHost(p.h_items);
    p.h_items = nullptr;
    p.h_items_cap = 0;
    if (cudaHostAlloc(reinterpret_cast<void**>(&p.h_items), sizeof(vitfe_item) * (size_t)n_items,
                      cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      return VITFE_ENOMEM;
    }
    p.h_items_cap = (size_t)n_items;
  }
  if ((size_t)(3 * nch) > p.h_small_cap) {
    if (p.h_small) cudaFreeHost(p.h_small);
    p.h_small = nullptr;
    p.h_small_cap = 0;
    if (cudaHostAlloc(reinterpret_cast<void**>(&p.h_small), sizeof(int32_t) * 3 * (size_t)nch,
                      cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      return VITFE_ENOMEM;
    }
    p.h_small_cap = 3 * (size_t)nch;
  }
  const float* tab = nullptr;
  if (vitfe::rope_table_for(c, head_dim, theta, p.comp, &tab) != cudaSuccess) return VITFE_ECUDA;
  // per-chunk descriptors (offsets relative to the chunk's pixel base) and statuses, kept
  // until the pipeline drains
  vitfe_item* chunk_items = p.h_items;
  int32_t* counts = p.h_small;
  int32_t* stat = p.h_small + nch;
  for (int k = 0; k < 2 * nch; ++k) stat[k] = 0;
  const int hh = head_dim / 2;
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < nch && e == cudaSuccess; ++k) {
    const int b = k & 1;
    const int i0 = cut[k], ni = cut[k + 1] - i0;
    const int64_t r0 = row0[i0], nr = row0[cut[k + 1]] - r0;
    for (int i = 0; i < ni; ++i) {
      chunk_items[(size_t)(i0 + i)] = items[i0 + i];
      chunk_items[(size_t)(i0 + i)].pixel_offset -= base[k];
    }
    counts[(size_t)k] = ni;
    // upload, once this staging set's previous download has finished
    e = cudaStreamWaitEvent(p.h2d, p.down[b], 0);
    if (e == cudaSuccess && span[k] > 0)
      e = cudaMemcpyAsync(p.px[b], pixels + base[k], (size_t)span[k], cudaMemcpyHostToDevice, p.h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(p.items[b], chunk_items + i0, sizeof(vitfe_item) * (size_t)ni,
                          cudaMemcpyHostToDevice, p.h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(p.n[b], counts + k, sizeof(int32_t), cudaMemcpyHostToDevice, p.h2d);
    if (e == cudaSuccess) e = cudaEventRecord(p.up[b], p.h2d);
    // the fused launch
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.comp, p.up[b], 0);
    if (e == cudaSuccess)
      e = vitfe::launch_embed(c, p.px[b], span[k], p.items[b], p.n[b], VITFE_MAX_ITEMS, nr, p.out[b], p.status[b],
                              p.comp, tab, head_dim / 4, p.cos[b], p.sin[b]);
    if (e == cudaSuccess) e = cudaEventRecord(p.done[b], p.comp);
    // download
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.d2h, p.done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<__nv_bfloat16*>(out) + (size_t)r0 * c.N, p.out[b],
                          (size_t)nr * c.N * sizeof(__nv_bfloat16), cudaMemcpyDeviceToHost, p.d2h);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(cos + (size_t)r0 * hh, p.cos[b], (size_t)nr * hh * sizeof(float), cudaMemcpyDeviceToHost,
                          p.d2h);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(sin + (size_t)r0 * hh, p.sin[b], (size_t)nr * hh * sizeof(float), cudaMemcpyDeviceToHost,
                          p.d2h);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(stat + 2 * k, p.status[b], 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, p.d2h);
    if (e == cudaSuccess) e = cudaEventRecord(p.down[b], p.d2h);
  }
  // drain every stream of the pipeline (also after an error: staging may not be reused early)
  const cudaError_t e1 = cudaStreamSynchronize(p.h2d);
  const cudaError_t e2 = cudaStreamSynchronize(p.comp);
  const cudaError_t e3 = cudaStreamSynchronize(p.d2h);
  if (e != cudaSuccess || e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) return VITFE_ECUDA;
  if (status != nullptr) {
    for (int k = 0; k < nch; ++k)
      if (stat[2 * (size_t)k] != 0) {
        status[0] = stat[2 * (size_t)k];
        status[1] = stat[2 * (size_t)k + 1] >= 0 ? stat[2 * (size_t)k + 1] + cut[k] : -1;
        break;
      }
  }
  return VITFE_OK;
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
