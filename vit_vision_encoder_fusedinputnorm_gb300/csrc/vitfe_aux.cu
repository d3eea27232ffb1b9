// Side paths of the front end (sm_103a): position ids, 2D-RoPE tables, standalone
// FusedInputNorm + patchify, and the create-time weight permutation.
#include <cmath>
#include <mutex>

#include "vitfe_internal.cuh"

namespace vitfe {
namespace {

constexpr int kAuxThreads = 256;

struct SmemTab {
  TabHdr hdr;
  uint32_t bad[kMaxItems / 32];
  uint32_t still[kMaxItems / 32];
  int start[kMaxItems + 1];
  __device__ ItemTab tab() { return ItemTab{start, bad, still, &hdr}; }
};

// Row -> (hpos, wpos) or (-1, -1) for pad rows and rows of invalid items.
__device__ __forceinline__ int2 row_pos(int r, SmemTab& t, const vitfe_item* items, int M) {
  int2 v = make_int2(-1, -1);
  if (r < t.hdr.live) {
    const int i = find_item(t.start, t.hdr.n, r);
    if (!tab_bit(t.bad, i)) {
      const int h = items[i].h, w = items[i].w;
      int tg, hh, ww;
      decode_local(r - t.start[i], h, w, M, tg, hh, ww);
      v = make_int2(hh, ww);
    }
  }
  return v;
}

// ---------------------------------------------------------------------------
// position ids ("vLLM 多模态推理｜ViT 性能优化" §3.3 step 2)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAuxThreads) pos_ids_kernel(const vitfe_item* items, const int32_t* n_items,
                                                              int max_items, int T, int M, int rows,
                                                              int2* pos, int32_t* status) {
  __shared__ SmemTab st;
  if (threadIdx.x < 32)
    build_item_table(items, n_items, max_items, -1, 1, T, M, rows, 0x7fffffff, st.tab());
  __syncthreads();
  write_status(status, &st.hdr);
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x)
    pos[r] = row_pos(r, st, items, M);
}

// ---------------------------------------------------------------------------
// 2D-RoPE ("vLLM 多模态推理｜ViT 性能优化" §3.3 steps 1, 3, 5)
// ---------------------------------------------------------------------------
// Axis table: tab[0][p][i] = cos(p * w_i), tab[1][p][i] = sin(p * w_i), w_i = theta^(-2i/d),
// d = head_dim / 2, i < nf = head_dim / 4, p < max(h, w) over the call's items.
// Angles and cos/sin in fp64, rounded once to fp32.
__global__ void __launch_bounds__(kAuxThreads) rope_table_kernel(const vitfe_item* items, const int32_t* n_items,
                                                                 int max_items, int T, int M, int rows,
                                                                 int nf, double theta, float* tab) {
  __shared__ SmemTab st;
  if (threadIdx.x < 32)
    build_item_table(items, n_items, max_items, -1, 1, T, M, rows, VITFE_ROPE_MAX_SIDE, st.tab());
  __syncthreads();
  const int maxside = st.hdr.maxside;
  const double d = 2.0 * nf;
  const int total = maxside * nf;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const int p = idx / nf;
    const int i = idx - p * nf;
    const double w = pow(theta, -2.0 * (double)i / d);
    double s, c;
    sincos((double)p * w, &s, &c);
    tab[(size_t)p * nf + i] = (float)c;
    tab[(size_t)VITFE_ROPE_MAX_SIDE * nf + (size_t)p * nf + i] = (float)s;
  }
}

// Expand: cos[r] = [tab_cos[hpos][0..nf) || tab_cos[wpos][0..nf)], sin likewise; pad rows (1, 0).
// One warp writes 32 consecutive rows as contiguous float4 stores.
__global__ void __launch_bounds__(kAuxThreads) rope_expand_kernel(const vitfe_item* items, const int32_t* n_items,
                                                                  int max_items, int T, int M, int rows,
                                                                  int nf, const float* __restrict__ tab,
                                                                  float* __restrict__ cosout,
                                                                  float* __restrict__ sinout, int32_t* status) {
  __shared__ SmemTab st;
  if (threadIdx.x < 32)
    build_item_table(items, n_items, max_items, -1, 1, T, M, rows, VITFE_ROPE_MAX_SIDE, st.tab());
  __syncthreads();
  write_status(status, &st.hdr);
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int width = 2 * nf;          // floats per row
  const int nvec = width >> 2;       // float4 per row
  const float* tc = tab;
  const float* ts = tab + (size_t)VITFE_ROPE_MAX_SIDE * nf;
  for (int wbase = (blockIdx.x * wpb + (threadIdx.x >> 5)) * 32; wbase < rows; wbase += gridDim.x * wpb * 32) {
    const int2 mypos = row_pos(wbase + lane, st, items, M);
    const int cnt = min(32, rows - wbase);
    const int total = cnt * nvec;
    const int iters = (total + 31) >> 5;
    float4* cdst = reinterpret_cast<float4*>(cosout + (size_t)wbase * width);
    float4* sdst = reinterpret_cast<float4*>(sinout + (size_t)wbase * width);
    for (int it = 0; it < iters; ++it) {
      const int f = it * 32 + lane;
      const int rr = min(f / nvec, 31);
      const int hp = __shfl_sync(0xffffffffu, mypos.x, rr);
      const int wp = __shfl_sync(0xffffffffu, mypos.y, rr);
      if (f < total) {
        const int cv = f - rr * nvec;
        float cvals[4], svals[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = 4 * cv + e;
          if (hp < 0) {
            cvals[e] = 1.0f;
            svals[e] = 0.0f;
          } else {
            const int p = col < nf ? hp : wp;
            const int i = col < nf ? col : col - nf;
            cvals[e] = __ldg(tc + (size_t)p * nf + i);
            svals[e] = __ldg(ts + (size_t)p * nf + i);
          }
        }
        __stcs(cdst + f, make_float4(cvals[0], cvals[1], cvals[2], cvals[3]));
        __stcs(sdst + f, make_float4(svals[0], svals[1], svals[2], svals[3]));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// standalone FusedInputNorm + patchify ("PR #55370 完整报告" 实现拆解 item 2;
// "vLLM 多模态推理｜ViT 性能优化" §2.2, §3.2): bf16 [rows][K], features (C, T, P, P).
// A CTA stages the pixel runs of RB rows in shared memory (aligned 4-byte loads),
// then writes the rows as contiguous 16-byte chunks.
// ---------------------------------------------------------------------------
constexpr int kRB = 32;

struct NpArgs {
  const uint8_t* pixels;
  int64_t pixel_bytes;
  const vitfe_item* items;
  const int32_t* n_items;
  int max_items;
  int rows;
  __nv_bfloat16* out;
  int32_t* status;
  float sc0, sc1, sc2, sh0, sh1, sh2;
  int P, T, M, K;
  int nwr;   // words per staged run
};

__global__ void __launch_bounds__(kAuxThreads) normalize_patchify_kernel(const NpArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  SmemTab& st = *reinterpret_cast<SmemTab*>(smem);
  size_t off = (sizeof(SmemTab) + 15) & ~size_t(15);
  int* kmap = reinterpret_cast<int*>(smem + off);
  off += ((size_t)a.K * 4 + 15) & ~size_t(15);
  const uint8_t** rbase = reinterpret_cast<const uint8_t**>(smem + off);
  off += kRB * sizeof(void*);
  int64_t* rrs = reinterpret_cast<int64_t*>(smem + off);
  off += kRB * sizeof(int64_t);
  int64_t* rfs = reinterpret_cast<int64_t*>(smem + off);
  off += kRB * sizeof(int64_t);
  int* rflag = reinterpret_cast<int*>(smem + off);   // bit0 valid, bit1 still
  off += kRB * sizeof(int);
  off = (off + 15) & ~size_t(15);
  uint32_t* raw = reinterpret_cast<uint32_t*>(smem + off);       // [kRB][T][P][nwr]
  off += (size_t)kRB * a.T * a.P * a.nwr * 4;
  uint8_t* rshift = smem + off;                                  // [kRB][T][P]

  if (threadIdx.x < 32)
    build_item_table(a.items, a.n_items, a.max_items, a.pixel_bytes, a.P, a.T, a.M, a.rows, 0x7fffffff, st.tab());
  const int PP = a.P * a.P, TPP = a.T * PP, RUN = 3 * a.P;
  for (int k = threadIdx.x; k < a.K; k += blockDim.x) {
    const int c = k / TPP;
    int rem = k - c * TPP;
    const int tt = rem / PP;
    rem -= tt * PP;
    const int ph = rem / a.P;
    const int pw = rem - ph * a.P;
    kmap[k] = (tt << 24) | (ph << 16) | ((pw * 3 + c) << 2) | c;
  }
  __syncthreads();
  write_status(a.status, &st.hdr);
  const float sc[3] = {a.sc0, a.sc1, a.sc2};
  const float sh[3] = {a.sh0, a.sh1, a.sh2};
  const int nchunk_row = (a.K % 8 == 0) ? a.K / 8 : 0;
  const int runs_per_row = a.T * a.P;

  for (int rb0 = blockIdx.x * kRB; rb0 < a.rows; rb0 += gridDim.x * kRB) {
    const int nrows = min(kRB, a.rows - rb0);
    if (threadIdx.x < kRB) {
      const int r = rb0 + threadIdx.x;
      int flag = 0;
      const uint8_t* b0 = nullptr;
      int64_t rs = 0, fs = 0;
      if (r < st.hdr.live) {
        const int i = find_item(st.start, st.hdr.n, r);
        if (!tab_bit(st.bad, i)) {
          const vitfe_item it = a.items[i];
          int tg, hh, ww;
          decode_local(r - st.start[i], it.h, it.w, a.M, tg, hh, ww);
          const int64_t H = (int64_t)it.h * a.P, W = (int64_t)it.w * a.P;
          const bool still = it.frames == 1;
          rs = W * 3;
          fs = still ? 0 : H * W * 3;
          const int64_t f0 = still ? 0 : (int64_t)tg * a.T;
          b0 = a.pixels + it.pixel_offset + ((f0 * H + (int64_t)hh * a.P) * W + (int64_t)ww * a.P) * 3;
          flag = 1 | (still ? 2 : 0);
        }
      }
      rbase[threadIdx.x] = b0;
      rrs[threadIdx.x] = rs;
      rfs[threadIdx.x] = fs;
      rflag[threadIdx.x] = flag;
    }
    __syncthreads();
    // stage pixel runs
    const int nword = nrows * runs_per_row * a.nwr;
    for (int idx = threadIdx.x; idx < nword; idx += blockDim.x) {
      const int row = idx / (runs_per_row * a.nwr);
      int rem = idx - row * runs_per_row * a.nwr;
      const int run = rem / a.nwr;
      const int w = rem - run * a.nwr;
      const int tt = run / a.P;
      const int ph = run - tt * a.P;
      const int flag = rflag[row];
      if (!(flag & 1) || (tt > 0 && (flag & 2))) continue;
      const uintptr_t addr = reinterpret_cast<uintptr_t>(rbase[row] + rfs[row] * tt + rrs[row] * ph);
      const uint32_t s = (uint32_t)(addr & 3u);
      if (w == 0) rshift[row * runs_per_row + run] = (uint8_t)s;
      if (4u * w < s + (uint32_t)RUN)
        raw[(size_t)(row * runs_per_row + run) * a.nwr + w] =
            __ldg(reinterpret_cast<const uint32_t*>(addr & ~uintptr_t(3)) + w);
    }
    __syncthreads();
    const uint8_t* rawb = reinterpret_cast<const uint8_t*>(raw);
    if (nchunk_row) {
      const int nch = nrows * nchunk_row;
      for (int idx = threadIdx.x; idx < nch; idx += blockDim.x) {
        const int row = idx / nchunk_row;
        const int q = idx - row * nchunk_row;
        const int flag = rflag[row];
        uint32_t pk[4] = {0u, 0u, 0u, 0u};
        if (flag & 1) {
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float x[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int m = kmap[8 * q + e + u];
              const int tt = (flag & 2) ? 0 : (m >> 24);
              const int run = tt * a.P + ((m >> 16) & 0xFF);
              const int bo = (m >> 2) & 0x3FFF;
              const int c = m & 3;
              const uint8_t v = rawb[(size_t)(row * runs_per_row + run) * a.nwr * 4 +
                                     rshift[row * runs_per_row + run] + bo];
              x[u] = fmaf((float)v, sc[c], sh[c]);
            }
            __nv_bfloat162 b2 = __floats2bfloat162_rn(x[0], x[1]);
            pk[e >> 1] = *reinterpret_cast<uint32_t*>(&b2);
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(a.out + (size_t)(rb0 + row) * a.K) + q;
        __stcs(dst, make_uint4(pk[0], pk[1], pk[2], pk[3]));
      }
    } else {
      const int nel = nrows * a.K;
      for (int idx = threadIdx.x; idx < nel; idx += blockDim.x) {
        const int row = idx / a.K;
        const int k = idx - row * a.K;
        const int flag = rflag[row];
        float x = 0.0f;
        if (flag & 1) {
          const int m = kmap[k];
          const int tt = (flag & 2) ? 0 : (m >> 24);
          const int run = tt * a.P + ((m >> 16) & 0xFF);
          const int c = m & 3;
          const uint8_t v = rawb[(size_t)(row * runs_per_row + run) * a.nwr * 4 +
                                 rshift[row * runs_per_row + run] + ((m >> 2) & 0x3FFF)];
          x = fmaf((float)v, sc[c], sh[c]);
        }
        a.out[(size_t)(rb0 + row) * a.K + k] = __float2bfloat16_rn(x);
      }
    }
    __syncthreads();
  }
}

size_t np_smem_bytes(int P, int T, int K, int nwr) {
  size_t off = (sizeof(SmemTab) + 15) & ~size_t(15);
  off += ((size_t)K * 4 + 15) & ~size_t(15);
  off += kRB * (sizeof(void*) + 2 * sizeof(int64_t) + sizeof(int));
  off = (off + 15) & ~size_t(15);
  off += (size_t)kRB * T * P * nwr * 4;
  off += (size_t)kRB * T * P;
  return off;
}

// ---------------------------------------------------------------------------
// create-time weight permutation: canonical (C, T, P, P) columns -> internal
// [slice t][(ph, pw, c)] columns, each slice zero-padded to kslice_pad.
// ---------------------------------------------------------------------------
__global__ void permute_weight_kernel(const __nv_bfloat16* __restrict__ W, const __nv_bfloat16* __restrict__ b,
                                      int N, int P, int T, int kslice, int kslice_pad,
                                      __nv_bfloat16* __restrict__ w_int, float* __restrict__ bias) {
  const int kint = T * kslice_pad;
  const int K = T * kslice;
  const long long total = (long long)N * kint;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(idx / kint);
    const int col = (int)(idx - (long long)n * kint);
    const int s = col / kslice_pad;
    const int kp = col - s * kslice_pad;
    __nv_bfloat16 v = __float2bfloat16_rn(0.0f);
    if (kp < kslice) {
      const int ph = kp / (3 * P);
      const int rem = kp - ph * 3 * P;
      const int pw = rem / 3;
      const int c = rem - pw * 3;
      const int k = ((c * T + s) * P + ph) * P + pw;
      v = W[(size_t)n * K + k];
    }
    w_int[idx] = v;
    if (col == 0) bias[n] = b ? __bfloat162float(b[n]) : 0.0f;
  }
}

int grid_for(long long work, int per_cta, int cap) {
  long long g = (work + per_cta - 1) / per_cta;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

}  // namespace

cudaError_t launch_pos_ids(const Ctx& c, const vitfe_item* items, const int32_t* n_items, int max_items,
                           int64_t rows, int32_t* pos, int32_t* status, cudaStream_t s) {
  const int grid = grid_for(rows, kAuxThreads, c.sm_count * 8);
  pos_ids_kernel<<<grid, kAuxThreads, 0, s>>>(items, n_items, max_items, c.T, c.M, (int)rows,
                                               reinterpret_cast<int2*>(pos), status);
  return cudaGetLastError();
}

cudaError_t launch_rope(const Ctx& c, const vitfe_item* items, const int32_t* n_items, int max_items,
                        int64_t rows, int head_dim, float theta, float* cos, float* sin, int32_t* status,
                        cudaStream_t s) {
  const int nf = head_dim / 4;
  rope_table_kernel<<<32, kAuxThreads, 0, s>>>(items, n_items, max_items, c.T, c.M, (int)rows, nf,
                                               (double)theta, c.rope_tab);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid = grid_for(rows, kAuxThreads, c.sm_count * 16);   // 8 warps x 32 rows per CTA
  rope_expand_kernel<<<grid, kAuxThreads, 0, s>>>(items, n_items, max_items, c.T, c.M, (int)rows, nf,
                                                  c.rope_tab, cos, sin, status);
  return cudaGetLastError();
}

cudaError_t launch_normalize_patchify(const Ctx& c, const uint8_t* pixels, int64_t pixel_bytes,
                                      const vitfe_item* items, const int32_t* n_items, int max_items,
                                      int64_t rows, void* out, int32_t* status, cudaStream_t s) {
  NpArgs a;
  a.pixels = pixels;
  a.pixel_bytes = pixel_bytes;
  a.items = items;
  a.n_items = n_items;
  a.max_items = max_items;
  a.rows = (int)rows;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.sc0 = c.scale[0]; a.sc1 = c.scale[1]; a.sc2 = c.scale[2];
  a.sh0 = c.shift[0]; a.sh1 = c.shift[1]; a.sh2 = c.shift[2];
  a.P = c.P;
  a.T = c.T;
  a.M = c.M;
  a.K = c.K;
  a.nwr = (3 * c.P + 3) / 4 + 1;
  const size_t smem = np_smem_bytes(c.P, c.T, c.K, a.nwr);
  cudaError_t e = cudaFuncSetAttribute(normalize_patchify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_for(rows, kRB, c.sm_count * 8);
  normalize_patchify_kernel<<<grid, kAuxThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_permute_weight(const Ctx& c, const __nv_bfloat16* W, const __nv_bfloat16* b, cudaStream_t s) {
  const long long total = (long long)c.N * c.kint;
  const int grid = grid_for(total, 256, c.sm_count * 16);
  permute_weight_kernel<<<grid, 256, 0, s>>>(W, b, c.N, c.P, c.T, c.kslice, c.kslice_pad, c.w_int, c.bias);
  return cudaGetLastError();
}

}  // namespace vitfe

// ---------------------------------------------------------------------------
// Allocation-free RoPE entry point.
//
// Some callers cannot allocate device memory at all: code running under an
// allocator they do not own (a serving runtime whose memory pool is carved up in
// advance, or a CUDA-graph capture that must not allocate), or a host process
// that is forbidden to call cudaMalloc after start-up.  vitfe_rope needs a handle,
// and creating one allocates.  vitfe_rope_noalloc runs the same two RoPE kernels
// with their axis-table scratch in the file-scope array below instead: 1 MiB,
// enough for position tables up to VITFE_ROPE_MAX_SIDE positions and head_dim up
// to 128.  Every GPU that loads this library holds the array until the process
// exits.
// ---------------------------------------------------------------------------
namespace vitfe {
namespace {

constexpr int kStaticRopeMaxHeadDim = 128;
constexpr size_t kStaticRopeFloats = (size_t)2 * VITFE_ROPE_MAX_SIDE * (kStaticRopeMaxHeadDim / 4);

// Host code must never pass this symbol to a kernel: on the host it names a
// shadow variable, not device memory.  Its device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) float g_rope_scratch[kStaticRopeFloats];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float* g_scratch_ptr[kMaxDevices] = {};
int g_scratch_sms[kMaxDevices] = {};

// Looks up (once per device, with that device current) the device address of the
// scratch array and the SM count.
cudaError_t static_scratch(int dev, float** ptr, int* sms) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_rope_scratch);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_scratch_sms[dev] = n;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *ptr = g_scratch_ptr[dev];
  *sms = g_scratch_sms[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace vitfe

extern "C" vitfe_status vitfe_rope_noalloc(int tpatch, int merge, const vitfe_item* items,
                                           const int32_t* n_items, int32_t max_items, int64_t rows,
                                           int head_dim, float theta, float* cos, float* sin,
                                           int32_t* status, cudaStream_t stream) {
  if (items == nullptr || n_items == nullptr) return VITFE_EINVAL;
  if (tpatch < 1 || tpatch > 4 || merge < 1 || merge > 8) return VITFE_EINVAL;
  if (max_items < 0 || max_items > VITFE_MAX_ITEMS) return VITFE_EINVAL;
  if (rows < 0 || rows > 0x7fffffffLL - 1024) return VITFE_EINVAL;
  if (head_dim < 8 || (head_dim % 8) != 0 || head_dim > VITFE_ROPE_MAX_HEAD_DIM) return VITFE_EINVAL;
  if (head_dim > vitfe::kStaticRopeMaxHeadDim) return VITFE_EUNSUPPORTED;   // beyond the static scratch
  if (!std::isfinite(theta) || !(theta > 0.0f)) return VITFE_EINVAL;
  if (rows > 0 && (cos == nullptr || sin == nullptr)) return VITFE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(cos) & 15u) || (reinterpret_cast<uintptr_t>(sin) & 15u)) return VITFE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(items) & 7u) || (reinterpret_cast<uintptr_t>(n_items) & 3u)) return VITFE_EINVAL;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return VITFE_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= vitfe::kMaxDevices) return VITFE_ECUDA;
  float* tab = nullptr;
  int sms = 0;
  if (vitfe::static_scratch(dev, &tab, &sms) != cudaSuccess) return VITFE_ECUDA;
  const int nf = head_dim / 4;
  vitfe::rope_table_kernel<<<32, vitfe::kAuxThreads, 0, stream>>>(items, n_items, max_items, tpatch, merge,
                                                                  (int)rows, nf, (double)theta, tab);
  if (cudaGetLastError() != cudaSuccess) return VITFE_ECUDA;
  const int grid = vitfe::grid_for(rows, vitfe::kAuxThreads, sms * 16);
  vitfe::rope_expand_kernel<<<grid, vitfe::kAuxThreads, 0, stream>>>(items, n_items, max_items, tpatch, merge,
                                                                     (int)rows, nf, tab, cos, sin, status);
  return cudaGetLastError() == cudaSuccess ? VITFE_OK : VITFE_ECUDA;
}
