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
// RoPE applied to Q/K ("vLLM 多模态推理｜ViT 性能优化" §3.3 step 6), rotate-half form:
// per head, feature i and feature i + hh (hh = head_dim / 2) rotate as one pair by the
// angle of table column i:  y[i] = x[i] c - x[i+hh] s,  y[i+hh] = x[i+hh] c + x[i] s,
// c = cos[r][i], s = sin[r][i]; fp32 arithmetic, bf16 round-to-nearest-even, in place.
// One warp per row at a time; lane units are (head, group of V pairs) of the row, Q heads
// first, walked without division.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bf16x4_to_f32(uint2 v, float* f) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
}
__device__ __forceinline__ uint2 f32_to_bf16x4(const float* f) {
  __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
  return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

// V pairs of one head half (V = 4: 8-byte accesses, V = 8: 16-byte accesses).
template <int V>
struct ApplyVec;
template <>
struct ApplyVec<4> {
  using X = uint2;
  __device__ static void load_tab(const float* p, float* f) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ static void unpack(X v, float* f) { bf16x4_to_f32(v, f); }
  __device__ static X pack(const float* f) { return f32_to_bf16x4(f); }
};
template <>
struct ApplyVec<8> {
  using X = uint4;
  __device__ static void load_tab(const float* p, float* f) {
    ApplyVec<4>::load_tab(p, f);
    ApplyVec<4>::load_tab(p + 4, f + 4);
  }
  __device__ static void unpack(X v, float* f) {
    bf16x4_to_f32(make_uint2(v.x, v.y), f);
    bf16x4_to_f32(make_uint2(v.z, v.w), f + 4);
  }
  __device__ static X pack(const float* f) {
    const uint2 a = f32_to_bf16x4(f), b = f32_to_bf16x4(f + 4);
    return make_uint4(a.x, a.y, b.x, b.y);
  }
};

// Lane units are (head, group of V pairs); each lane takes NB units per step (u, u + 32,
// ...) and issues all their Q/K loads before any table load or arithmetic.
template <int V, int NB>
__global__ void __launch_bounds__(kAuxThreads) rope_apply_kernel(const float* __restrict__ cos,
                                                                 const float* __restrict__ sin, int rows, int hh,
                                                                 int heads_q, int heads_k, __nv_bfloat16* q,
                                                                 long long q_stride, __nv_bfloat16* k,
                                                                 long long k_stride) {
  using AV = ApplyVec<V>;
  using X = typename AV::X;
  const int lane = threadIdx.x & 31;
  const int gw = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  const int nw = (int)((gridDim.x * (unsigned)blockDim.x) >> 5);
  const int G = hh / V;                        // groups of V pairs per head
  const int units = (heads_q + heads_k) * G;   // per row
  const int h0 = lane / G, j0 = lane - h0 * G;
  const int dh = 32 / G, dj = 32 - dh * G;     // a step of 32 units in (head, group)
  for (int r = gw; r < rows; r += nw) {
    const float* cr = cos + (size_t)r * hh;
    const float* sr = sin + (size_t)r * hh;
    __nv_bfloat16* qr = q + (size_t)r * q_stride;
    __nv_bfloat16* kr = k + (size_t)r * k_stride;
    int hd = h0, j = j0;
    for (int u = lane; u < units; u += 32 * NB) {
      X* p1[NB];
      X* p2[NB];
      int jj[NB];
      X v1[NB], v2[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const bool live = u + 32 * b < units;
        __nv_bfloat16* x = (hd < heads_q) ? qr + (size_t)hd * (2 * hh) : kr + (size_t)(hd - heads_q) * (2 * hh);
        p1[b] = reinterpret_cast<X*>(x + V * j);
        p2[b] = reinterpret_cast<X*>(x + hh + V * j);
        jj[b] = j;
        if (live) {
          v1[b] = *p1[b];
          v2[b] = *p2[b];
          hd += dh;
          j += dj;
          if (j >= G) {
            j -= G;
            ++hd;
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (u + 32 * b >= units) break;
        float c[V], sn[V], a1[V], a2[V], y1[V], y2[V];
        AV::load_tab(cr + V * jj[b], c);
        AV::load_tab(sr + V * jj[b], sn);
        AV::unpack(v1[b], a1);
        AV::unpack(v2[b], a2);
#pragma unroll
        for (int e = 0; e < V; ++e) {
          y1[e] = fmaf(a1[e], c[e], -(a2[e] * sn[e]));
          y2[e] = fmaf(a2[e], c[e], a1[e] * sn[e]);
        }
        *p1[b] = AV::pack(y1);
        *p2[b] = AV::pack(y2);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Attention sequence boundaries ("vLLM 多模态推理｜ViT 性能优化" §3.4): the encoder's
// attention keeps each image apart, so its varlen kernels take the first row of every
// sequence.  The encoder sees single images and single frames (§3.3), so each temporal
// group of an item is one sequence of h*w rows: cu[0] = 0 and, item by item and group by
// group, cu[s + 1] = cu[s] + h*w, clipped to the bucket (a sequence past it is dropped).
// Entries past the last sequence, up to max_seqs, repeat the last boundary; info =
// {number of sequences, longest sequence}.  More than max_seqs sequences: the first
// max_seqs are written and the status word reports VITFE_EDEVICE_RANGE.
// One CTA: warp 0 builds the item table, the CTA scans the items' sequence counts.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAuxThreads) cu_seqlens_kernel(const vitfe_item* items, const int32_t* n_items,
                                                                 int max_items, int T, int M, int rows,
                                                                 int max_seqs, int32_t* cu, int32_t* info,
                                                                 int32_t* status) {
  __shared__ SmemTab st;
  __shared__ int sbase[kMaxItems + 1];    // first sequence of each item
  __shared__ int smax[kAuxThreads / 32];
  if (threadIdx.x < 32)
    build_item_table(items, n_items, max_items, -1, 1, T, M, rows, 0x7fffffff, st.tab());
  __syncthreads();
  const int n = st.hdr.n;
  // sequences of item i: its temporal groups whose rows start inside the bucket
  auto nseq_of = [&](int i) -> int {
    const int hw = items[i].h * items[i].w;
    const int r0 = st.start[i], r1 = st.start[i + 1];
    if (hw <= 0 || r1 <= r0) return 0;
    return (r1 - r0 + hw - 1) / hw;
  };
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < n; ++i) {
      sbase[i] = acc;
      acc += nseq_of(i);
    }
    sbase[n] = acc;
  }
  __syncthreads();
  const int total = sbase[n];
  const int nw = min(total, max_seqs);
  int mx = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int hw = items[i].h * items[i].w;
    const int k = nseq_of(i);
    for (int g = 0; g < k; ++g) {
      const int sidx = sbase[i] + g;
      const int end = min(st.start[i] + (g + 1) * hw, st.start[i + 1]);
      mx = max(mx, end - (st.start[i] + g * hw));
      if (sidx < nw) cu[sidx + 1] = end;
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
  if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = mx;
  __syncthreads();
  // pad: entries past the last boundary repeat it (only when every sequence fitted, so the
  // last boundary is the end of the live rows)
  const int last = (nw == 0) ? 0 : st.hdr.live;
  for (int k = nw + 1 + threadIdx.x; k <= max_seqs; k += blockDim.x) cu[k] = last;
  if (threadIdx.x == 0) {
    cu[0] = 0;
    int m = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, smax[w]);
    info[0] = nw;
    info[1] = m;
    if (status != nullptr) {
      if (st.hdr.code == kOk && total > max_seqs) {
        status[0] = kRange;
        status[1] = -1;
      } else {
        status[0] = st.hdr.code;
        status[1] = st.hdr.bad_item;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 2D-RoPE ("vLLM 多模态推理｜ViT 性能优化" §3.3 steps 1, 3, 5)
// ---------------------------------------------------------------------------
__device__ void rope_fill(float* tab, int nf, double theta, int maxside);

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
  rope_fill(tab, nf, theta, maxside);
}

// Every position of the table: the handle's cos/sin cache, built once per (head_dim, theta).
__global__ void __launch_bounds__(kAuxThreads) rope_cache_kernel(int nf, double theta, float* tab) {
  rope_fill(tab, nf, theta, VITFE_ROPE_MAX_SIDE);
}

__device__ void rope_fill(float* tab, int nf, double theta, int maxside) {
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
  const bool vec_tab = (nf % 4) == 0;   // table rows 16-byte aligned, halves whole float4 groups
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
        float4 cvv, svv;
        if (hp < 0) {
          cvv = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
          svv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        } else if (vec_tab) {
          // each group of 4 columns lies in one half: one 16-byte load per table
          const int col = 4 * cv;
          const int p = col < nf ? hp : wp;
          const int i = col < nf ? col : col - nf;
          cvv = __ldg(reinterpret_cast<const float4*>(tc + (size_t)p * nf + i));
          svv = __ldg(reinterpret_cast<const float4*>(ts + (size_t)p * nf + i));
        } else {
          float cvals[4], svals[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = 4 * cv + e;
            const int p = col < nf ? hp : wp;
            const int i = col < nf ? col : col - nf;
            cvals[e] = __ldg(tc + (size_t)p * nf + i);
            svals[e] = __ldg(ts + (size_t)p * nf + i);
          }
          cvv = make_float4(cvals[0], cvals[1], cvals[2], cvals[3]);
          svv = make_float4(svals[0], svals[1], svals[2], svals[3]);
        }
        __stcs(cdst + f, cvv);
        __stcs(sdst + f, svv);
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

// Specialised for patch P (14, 16) and tpatch T (1, 2).  Each warp owns two output rows at
// a time, end to end: lanes 0-1 decode the rows, one lane per (row, pixel row ph) loads the
// 3P-byte run of each stored frame once (aligned 4-byte loads) and writes, for every channel
// c and temporal slice t, the P features (c, t, ph, 0..P-1) of the canonical order into the
// warp's shared-memory copy of the two rows, which the TMA engine then writes out with one
// bulk copy per row (keeping the copy-out off the load/store pipe, which the pixel loads
// and stage writes keep busy).  The loads of the warp's next pair are issued before the
// current pair is converted, so every warp keeps one pair of pixel runs in flight while it
// converts; there is no CTA-wide barrier in the loop.
constexpr int kNpWarpRows = 2;

// Two fp32 lanes in one 64-bit register (packed f32x2 arithmetic, exact per lane).
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, uint32_t& lo, uint32_t& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
// x = (v - 2^23) * scale + shift on both lanes; v holds 2^23 + byte (exact).
__device__ __forceinline__ uint64_t norm2(uint64_t v, uint64_t scale2, uint64_t shift2) {
  const uint64_t m = 0xCB000000CB000000ull;   // (-2^23, -2^23)
  uint64_t t, x;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(v), "l"(m));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x) : "l"(t), "l"(scale2), "l"(shift2));
  return x;
}

// Stage row stride (32-bit words): the features (c, t, ph, pw..pw+1) of lane (row, ph) sit
// at row * RS + ((c * T + t) * P + ph) * P / 2 + pw / 2, so one store instruction touches
// banks (P/2) * ph + RS * row (mod 32).  For P = 14 the 14 banks of one row are distinct and
// RS = 16 (mod 32) keeps the second row's 14 off them; for P = 16 a row covers 4 banks and
// RS = 4 (mod 32) at least keeps the rows apart.  RS stays a multiple of 4 (16-byte reads).
__host__ __device__ constexpr int np_stage_rs(int P, int KW) {
  return KW + ((((P == 14) ? 16 : 4) - KW % 32) + 32) % 32;
}

template <int P, int T>
struct NpPair {
  static constexpr int RUN = 3 * P;                 // bytes of one pixel row of one patch
  // aligned chunks of CB bytes covering it: 16 when runs start on 16-byte bounds in the
  // usual layout (3P a multiple of 16), else 8 (fewer selects to realign scattered runs)
  static constexpr int CB = (RUN % 16 == 0) ? 16 : 8;
  static constexpr int NC = (RUN + CB - 1 + CB - 1) / CB;
  static constexpr int NWR = NC * CB / 4;           // words held
  uint32_t raw[T][NWR];
  uint32_t sft[T];                                  // byte offset of the run in raw[t][0] (< CB)
  int flag;                                         // bit 0: row valid, bit 1: still item
  int nrows;                                        // rows of this pair inside [0, rows)
};

// Decode rows rb, rb + 1 and issue this lane's loads (lane = row * P + ph).
template <int P, int T>
__device__ __forceinline__ void np_fetch(NpPair<P, T>& q, const NpArgs& a, const SmemTab& st, int rb,
                                         int lane) {
  q.nrows = min(kNpWarpRows, a.rows - rb);
  int flag = 0;
  unsigned long long b0 = 0ull;
  long long rs = 0, fs = 0;
  if (lane < q.nrows) {
    const int r = rb + lane;
    if (r < st.hdr.live) {
      const int i = find_item(st.start, st.hdr.n, r);
      if (!tab_bit(st.bad, i)) {
        const vitfe_item it = a.items[i];
        int tg, hh, ww;
        decode_local(r - st.start[i], it.h, it.w, a.M, tg, hh, ww);
        const int64_t H = (int64_t)it.h * P, W = (int64_t)it.w * P;
        const bool still = it.frames == 1;
        rs = W * 3;
        fs = still ? 0 : H * W * 3;
        const int64_t f0 = still ? 0 : (int64_t)tg * T;
        b0 = reinterpret_cast<unsigned long long>(a.pixels + it.pixel_offset +
                                                  ((f0 * H + (int64_t)hh * P) * W + (int64_t)ww * P) * 3);
        flag = 1 | (still ? 2 : 0);
      }
    }
  }
  const int lr = lane / P;
  const int ph = lane - lr * P;
  q.flag = __shfl_sync(0xffffffffu, flag, lr);
  const unsigned long long base = __shfl_sync(0xffffffffu, b0, lr);
  const long long mrs = __shfl_sync(0xffffffffu, rs, lr);
  const long long mfs = __shfl_sync(0xffffffffu, fs, lr);
  if (lr >= q.nrows) q.flag = 0;
  const uintptr_t addr0 = (uintptr_t)(base + (unsigned long long)(mrs * ph));
#pragma unroll
  for (int tt = 0; tt < T; ++tt) {
    // a still's one frame serves every temporal slice: load it once.  8-byte loads (each
    // chunk holds a byte of the run, so none leaves the buffer): half the load instructions
    // of 4-byte ones on the load/store pipe that bounds this kernel
    const bool ld = (q.flag & 1) && (tt == 0 || !(q.flag & 2));
    constexpr int CB = NpPair<P, T>::CB;
    const uintptr_t at = addr0 + (uintptr_t)(mfs * tt);
    q.sft[tt] = (uint32_t)(at & (CB - 1));
#pragma unroll
    for (int c = 0; c < NpPair<P, T>::NC; ++c) {
      const bool hit = ld && (uint32_t)(CB * c) < q.sft[tt] + NpPair<P, T>::RUN;
      if constexpr (CB == 16) {
        const uint4* c0 = reinterpret_cast<const uint4*>(at & ~uintptr_t(15));
        const uint4 v = hit ? __ldg(c0 + c) : make_uint4(0u, 0u, 0u, 0u);
        q.raw[tt][4 * c] = v.x;
        q.raw[tt][4 * c + 1] = v.y;
        q.raw[tt][4 * c + 2] = v.z;
        q.raw[tt][4 * c + 3] = v.w;
      } else {
        const uint2* c0 = reinterpret_cast<const uint2*>(at & ~uintptr_t(7));
        const uint2 v = hit ? __ldg(c0 + c) : make_uint2(0u, 0u);
        q.raw[tt][2 * c] = v.x;
        q.raw[tt][2 * c + 1] = v.y;
      }
    }
  }
}

// Convert this lane's runs into the stage (row lr, pixel row ph).
template <int P, int T>
__device__ __forceinline__ void np_convert(const NpPair<P, T>& q, uint32_t* srow, int ph, const float* sc,
                                           const float* sh) {
  constexpr int NA = (3 * P + 3) / 4;
  const bool valid = q.flag & 1;
  const bool still = q.flag & 2;
  constexpr int WMAX = NpPair<P, T>::CB / 4 - 1;   // largest word offset of a run in its chunks
  static_assert(NA + WMAX < NpPair<P, T>::NWR, "the 4-byte view of a run lies inside its chunks");
#pragma unroll
  for (int tt = 0; tt < T; ++tt) {
    if (tt > 0 && still) break;
    const uint32_t sel = 0x3210u + 0x1111u * (q.sft[tt] & 3u);
    // the run's aligned words start wo words into the chunks: v[k] = raw[wo + k]
    const uint32_t wo = q.sft[tt] >> 2;
    uint32_t v[NA + 1];
#pragma unroll
    for (int k = 0; k <= NA; ++k) {
      const uint32_t a01 = (wo & 1u) ? q.raw[tt][k + 1] : q.raw[tt][k];
      if constexpr (WMAX >= 2) {
        const uint32_t a23 = (wo & 1u) ? q.raw[tt][k + 3] : q.raw[tt][k + 2];
        v[k] = (wo & 2u) ? a23 : a01;
      } else {
        v[k] = a01;
      }
    }
    uint32_t al[NA];
#pragma unroll
    for (int w = 0; w < NA; ++w) al[w] = __byte_perm(v[w], v[w + 1], sel);
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const uint64_t s2 = pack2(__float_as_uint(sc[c]), __float_as_uint(sc[c]));
      const uint64_t h2 = pack2(__float_as_uint(sh[c]), __float_as_uint(sh[c]));
#pragma unroll
      for (int pw = 0; pw < P; pw += 2) {
        const int e0 = 3 * pw + c, e1 = 3 * (pw + 1) + c;
        const uint32_t v0 = __byte_perm(al[e0 >> 2], 0x4B000000u, 0x7540u + (e0 & 3));
        const uint32_t v1 = __byte_perm(al[e1 >> 2], 0x4B000000u, 0x7540u + (e1 & 3));
        uint32_t x0, x1;
        unpack2(norm2(pack2(v0, v1), s2, h2), x0, x1);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(x0), __uint_as_float(x1));
        const uint32_t word = valid ? *reinterpret_cast<uint32_t*>(&b2) : 0u;
        if (still) {
#pragma unroll
          for (int t2 = 0; t2 < T; ++t2) srow[(((c * T + t2) * P + ph) * P + pw) >> 1] = word;
        } else {
          srow[(((c * T + tt) * P + ph) * P + pw) >> 1] = word;
        }
      }
    }
  }
}

// Bulk asynchronous copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this CTA's shared memory to global memory, by the TMA engine.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed bulk store has finished reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed bulk store is complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int P, int T>
__global__ void __launch_bounds__(kAuxThreads, 3) normalize_patchify_p_kernel(const NpArgs a) {
  constexpr int KW = 3 * T * P * P / 2;                     // bf16 pairs per row
  constexpr int RS = np_stage_rs(P, KW);
  static_assert(KW % 4 == 0 && RS % 4 == 0, "16-byte rows");
  static_assert(kNpWarpRows * P <= 32, "one lane per (row, pixel row)");
  extern __shared__ __align__(16) uint8_t np_smem[];
  __shared__ SmemTab st;
  if (threadIdx.x < 32)
    build_item_table(a.items, a.n_items, a.max_items, a.pixel_bytes, P, a.T, a.M, a.rows, 0x7fffffff, st.tab());
  __syncthreads();
  write_status(a.status, &st.hdr);
  const float sc[3] = {a.sc0, a.sc1, a.sc2};
  const float sh[3] = {a.sh0, a.sh1, a.sh2};
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  uint32_t* stage = reinterpret_cast<uint32_t*>(np_smem) + (size_t)warp * (RS + KW);
  const int lr = lane / P;
  const int ph = lane - lr * P;
  const int step = gridDim.x * wpb * kNpWarpRows;
  int rb = (blockIdx.x * wpb + warp) * kNpWarpRows;
  if (rb >= a.rows) return;
  NpPair<P, T> cur;
  np_fetch<P, T>(cur, a, st, rb, lane);
  for (;;) {
    const int rn = rb + step;
    NpPair<P, T> nxt;
    if (rn < a.rows) np_fetch<P, T>(nxt, a, st, rn, lane);
    // the previous pair's bulk stores must have read the stage before it is rewritten
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    if (lr < cur.nrows) np_convert<P, T>(cur, stage + lr * RS, ph, sc, sh);
    // each row goes out as one bulk copy by the TMA engine, off the load/store pipe
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      for (int row = 0; row < cur.nrows; ++row)
        bulk_store(a.out + (size_t)(rb + row) * (2 * KW), stage + row * RS, (uint32_t)(KW * 4));
      bulk_commit();
    }
    if (rn >= a.rows) break;
    cur = nxt;
    rb = rn;
  }
  if (lane == 0) bulk_wait_all();
}

int grid_for(long long work, int per_cta, int cap) {
  long long g = (work + per_cta - 1) / per_cta;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

template <int P, int T>
constexpr size_t np_p_stage_bytes() {
  return (size_t)(kAuxThreads / 32) * (np_stage_rs(P, 3 * T * P * P / 2) + 3 * T * P * P / 2) * 4;
}

// Opt the specialised kernel of (P, T) into its stage size and record its resident CTAs per
// SM in the handle (its persistent grid is SMs x that).
template <int P, int T>
cudaError_t np_p_configure(Ctx& c) {
  const size_t stage_bytes = np_p_stage_bytes<P, T>();
  cudaError_t e = cudaFuncSetAttribute(normalize_patchify_p_kernel<P, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)stage_bytes);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, normalize_patchify_p_kernel<P, T>, kAuxThreads, stage_bytes);
  if (e != cudaSuccess) return e;
  c.np_per_sm = n > 0 ? n : 1;
  return cudaSuccess;
}

template <int P, int T>
cudaError_t launch_np_p(const Ctx& c, const NpArgs& a, cudaStream_t s) {
  const int grid = grid_for(a.rows, (kAuxThreads / 32) * kNpWarpRows, c.sm_count * c.np_per_sm);
  normalize_patchify_p_kernel<P, T><<<grid, kAuxThreads, np_p_stage_bytes<P, T>(), s>>>(a);
  return cudaGetLastError();
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
// Create-time weight tiling.  The embed kernel reads W as whole shared-memory images:
// block (pass p, CTA half r, temporal slice s, K block j) holds the bnh = bn/2 weight
// rows n = p*bn + r*(npw/2) + i (i < npw/2, npw = min(bn, N - p*bn); other rows zero)
// times the 64 internal features 64*j + e of slice s, in the 128-byte-swizzled K-major
// layout the MMA descriptor expects: row i at i*128, 16-byte chunk q of the row at
// chunk position q ^ (i & 7).  Internal feature kp of a slice is (ph*P + pw)*3 + c
// (zero past 3*P*P); it holds canonical column ((c*T + s)*P + ph)*P + pw.
// ---------------------------------------------------------------------------
//
// fold != 0 writes the folded-still weight instead: one slice whose feature holds the sum
// of the T temporal slices' weights, taken in double (exact) and rounded once to bf16.
__global__ void tile_weight_kernel(const __nv_bfloat16* __restrict__ W, const __nv_bfloat16* __restrict__ b,
                                   int N, int P, int T, int nblk, int bn, int fold,
                                   __nv_bfloat16* __restrict__ w_tile, float* __restrict__ bias) {
  const int kslice = 3 * P * P;
  const int K = T * kslice;
  const int bnh = bn / 2;
  const int npass = (N + bn - 1) / bn;
  const int TL = fold ? 1 : T;                 // slices in the layout
  const bool shared_tail = w_tail_shared(kslice);
  const int nfb = shared_tail ? kslice / 64 : nblk;   // blocks with one image per slice
  const int imgs = w_images(kslice, TL);              // images per (pass, CTA half)
  const long long per_blk = (long long)bnh * 64;
  const long long total = (long long)npass * 2 * imgs * per_blk;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long blk = idx / per_blk;
    const int within = (int)(idx - blk * per_blk);
    const int i = within >> 6;
    const int qp = (within >> 3) & 7;                 // physical chunk in the row
    const int e = ((qp ^ (i & 7)) << 3) | (within & 7);
    const int g = (int)(blk % imgs);
    const int r = (int)((blk / imgs) & 1);
    const int p = (int)(blk / ((long long)imgs * 2));
    const int npw = min(bn, N - p * bn);
    int sl, kp;
    bool inside;
    if (shared_tail && g == TL * nfb) {
      // the slices' tails: slice e / 16 at K16 offset e / 16
      sl = e >> 4;
      kp = 64 * nfb + (e & 15);
      inside = sl < TL && kp < kslice;
    } else {
      sl = g / nfb;
      kp = 64 * (g % nfb) + e;
      inside = kp < kslice;
    }
    __nv_bfloat16 v = __float2bfloat16_rn(0.0f);
    if (i < npw / 2 && inside) {
      const int n = p * bn + r * (npw / 2) + i;
      const int ph = kp / (3 * P);
      const int rem = kp - ph * 3 * P;
      const int pw = rem / 3;
      const int c = rem - pw * 3;
      if (fold) {
        double acc = 0.0;
        for (int s2 = 0; s2 < T; ++s2) acc += (double)__bfloat162float(W[(size_t)n * K + ((c * T + s2) * P + ph) * P + pw]);
        v = __double2bfloat16(acc);
      } else {
        v = W[(size_t)n * K + ((c * T + sl) * P + ph) * P + pw];
      }
    }
    w_tile[idx] = v;
  }
  if (fold) return;
  for (long long n = (long long)blockIdx.x * blockDim.x + threadIdx.x; n < N; n += (long long)gridDim.x * blockDim.x)
    bias[n] = b ? __bfloat162float(b[n]) : 0.0f;
}

}  // namespace

cudaError_t launch_pos_ids(const Ctx& c, const vitfe_item* items, const int32_t* n_items, int max_items,
                           int64_t rows, int32_t* pos, int32_t* status, cudaStream_t s) {
  const int grid = grid_for(rows, kAuxThreads, c.sm_count * 8);
  pos_ids_kernel<<<grid, kAuxThreads, 0, s>>>(items, n_items, max_items, c.T, c.M, (int)rows,
                                               reinterpret_cast<int2*>(pos), status);
  return cudaGetLastError();
}

cudaError_t launch_rope_apply(const float* cos, const float* sin, int64_t rows, int head_dim, void* q,
                              int heads_q, int64_t q_stride, void* k, int heads_k, int64_t k_stride,
                              cudaStream_t s) {
  if (rows == 0 || heads_q + heads_k == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int warps_per_cta = kAuxThreads / 32;
  const int grid = grid_for(rows, warps_per_cta, sms * 8);
  // 16-byte accesses when every head half and row start is 16-byte aligned
  const int hh = head_dim / 2;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool v8 = (hh % 8) == 0 && (heads_q == 0 || (a16(q) && q_stride % 8 == 0)) &&
                  (heads_k == 0 || (a16(k) && k_stride % 8 == 0));
  if (v8)
    rope_apply_kernel<8, 4><<<grid, kAuxThreads, 0, s>>>(cos, sin, (int)rows, hh, heads_q, heads_k,
                                                      static_cast<__nv_bfloat16*>(q), q_stride,
                                                      static_cast<__nv_bfloat16*>(k), k_stride);
  else
    rope_apply_kernel<4, 4><<<grid, kAuxThreads, 0, s>>>(cos, sin, (int)rows, hh, heads_q, heads_k,
                                                      static_cast<__nv_bfloat16*>(q), q_stride,
                                                      static_cast<__nv_bfloat16*>(k), k_stride);
  return cudaGetLastError();
}

cudaError_t launch_cu_seqlens(const Ctx& c, const vitfe_item* items, const int32_t* n_items, int max_items,
                              int64_t rows, int max_seqs, int32_t* cu, int32_t* info, int32_t* status,
                              cudaStream_t s) {
  cu_seqlens_kernel<<<1, kAuxThreads, 0, s>>>(items, n_items, max_items, c.T, c.M, (int)rows, max_seqs, cu, info,
                                              status);
  return cudaGetLastError();
}

cudaError_t rope_table_for(Ctx& c, int head_dim, float theta, cudaStream_t s, const float** tab_out) {
  const int nf = head_dim / 4;
  const size_t slot_floats = (size_t)2 * VITFE_ROPE_MAX_SIDE * (VITFE_ROPE_MAX_HEAD_DIM / 4);
  // the cos/sin table of this (head_dim, theta): built once over every position, then reused
  int slot = -1;
  for (int k = 0; k < c.rope_used; ++k)
    if (c.rope_hd[k] == head_dim && c.rope_theta[k] == theta) slot = k;
  if (slot < 0 && c.rope_used < Ctx::kRopeSlots) {
    slot = c.rope_used++;
    c.rope_hd[slot] = head_dim;
    c.rope_theta[slot] = theta;
    c.rope_built[slot] = false;
  }
  const bool transient = slot < 0;
  float* tab = c.rope_tab + (size_t)(transient ? Ctx::kRopeSlots : slot) * slot_floats;
  if (transient || !c.rope_built[slot]) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return e;
    rope_cache_kernel<<<grid_for((long long)VITFE_ROPE_MAX_SIDE * nf, kAuxThreads, c.sm_count * 4), kAuxThreads, 0,
                        s>>>(nf, (double)theta, tab);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!transient && cap == cudaStreamCaptureStatusNone) c.rope_built[slot] = true;
  }
  *tab_out = tab;
  return cudaSuccess;
}

cudaError_t launch_rope(Ctx& c, const vitfe_item* items, const int32_t* n_items, int max_items, int64_t rows,
                        int head_dim, float theta, float* cos, float* sin, int32_t* status, cudaStream_t s) {
  const int nf = head_dim / 4;
  const float* tab = nullptr;
  cudaError_t e = rope_table_for(c, head_dim, theta, s, &tab);
  if (e != cudaSuccess) return e;
  const int grid = grid_for(rows, kAuxThreads, c.sm_count * 16);   // 8 warps x 32 rows per CTA
  rope_expand_kernel<<<grid, kAuxThreads, 0, s>>>(items, n_items, max_items, c.T, c.M, (int)rows, nf, tab, cos, sin,
                                                  status);
  return cudaGetLastError();
}

cudaError_t np_configure(Ctx& c) {
  if (c.P == 14 && c.T == 2) return np_p_configure<14, 2>(c);
  if (c.P == 16 && c.T == 2) return np_p_configure<16, 2>(c);
  if (c.P == 16 && c.T == 1) return np_p_configure<16, 1>(c);
  return cudaSuccess;
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
  if (c.P == 14 && c.T == 2) return launch_np_p<14, 2>(c, a, s);
  if (c.P == 16 && c.T == 2) return launch_np_p<16, 2>(c, a, s);
  if (c.P == 16 && c.T == 1) return launch_np_p<16, 1>(c, a, s);
  const size_t smem = np_smem_bytes(c.P, c.T, c.K, a.nwr);
  cudaError_t e = cudaFuncSetAttribute(normalize_patchify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_for(rows, kRB, c.sm_count * 8);
  normalize_patchify_kernel<<<grid, kAuxThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_tile_weight(const Ctx& c, const __nv_bfloat16* W, const __nv_bfloat16* b, cudaStream_t s) {
  const long long total = (long long)c.w_tile_bytes / 2;
  const int grid = grid_for(total, 256, c.sm_count * 16);
  tile_weight_kernel<<<grid, 256, 0, s>>>(W, b, c.N, c.P, c.T, c.nblk, c.bn, 0, c.w_tile, c.bias);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || c.w_tile_f == nullptr) return e;
  const long long total_f = (long long)c.w_tile_f_bytes / 2;
  tile_weight_kernel<<<grid_for(total_f, 256, c.sm_count * 16), 256, 0, s>>>(W, b, c.N, c.P, c.T, c.nblk, c.bn, 1,
                                                                            c.w_tile_f, c.bias);
  return cudaGetLastError();
}

}  // namespace vitfe

// ---------------------------------------------------------------------------
// Allocation-free RoPE entry point.
//
// Some callers cannot allocate device memory at all: code running under an
// allocator they do not own (a serving runtime whose memory pool is carved up in
// advance), or a host process that is forbidden to call cudaMalloc after start-up,
// where an allocation can fail or stall the other work sharing the GPU.  vitfe_rope needs a handle,
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
