// Fused FusedInputNorm + merge-order patchify + patch-embed GEMM + bias (sm_103a).
//
// What it computes ("PR #55370 完整报告" 实现拆解 item 2; "vLLM 多模态推理｜ViT 性能优化"
// §2.2 and §3.2): for every patch row r (items in order, merge order inside an item)
//     out[r][n] = bf16( sum_k A[r][k] * W[n][k] + b[n] ),
//     A[r][k]   = bf16( v * rescale/std_c - mean_c/std_c ),
// where v is the uint8 pixel feature k of patch r.  A never reaches device memory.
//
// Structure (one persistent CTA per SM, 10 warps):
//   warps 0-3  A producers: one thread per tile row gathers uint8 pixel runs with
//              aligned 4-byte loads, normalises in fp32, rounds to bf16 and stores
//              into 128-byte-swizzled K-major shared-memory blocks (64 features each);
//   warp 8     TMA producer of W tiles (box 64 x bn, 128-byte swizzle);
//   warp 9     TMEM allocator and the single MMA-issuing thread (tcgen05.mma kind::f16,
//              M=128, N=bn, fp32 accumulators double-buffered in tensor memory);
//   warps 4-7  epilogue: tcgen05.ld of the accumulator, + bias, bf16 RNE, stores.
//
// Features inside one temporal slice are ordered (ph, pw, c) so that each patch row
// of pixels is one contiguous byte run; the weight was permuted the same way once
// at create.  The whole slice of A (all K blocks) stays resident in shared memory
// while the tile loops over the N passes; for stills the temporal slices are equal,
// so one resident slice feeds the MMAs of every slice ("resident" tiles).  Tiles
// holding video rows re-produce A per (pass, slice) ("stream" tiles).
//
// Every mbarrier wait is bounded (global timer); on expiry the CTA drains its async
// copies and MMAs, frees its tensor memory, writes VITFE_EDEVICE_TIMEOUT and exits.
#include "vitfe_internal.cuh"

namespace vitfe {
namespace {

constexpr int kThreads = 320;
constexpr int kProducerThreads = 128;
constexpr int kEpiWarp0 = 4;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kABlockBytes = kTileM * 128;   // 128 rows x 64 bf16

enum TileKind : int { kPad = 0, kResident = 1, kStream = 2 };

struct EmbedArgs {
  const uint8_t* pixels;
  int64_t pixel_bytes;
  const vitfe_item* items;
  const int32_t* n_items;
  int max_items;
  int rows;
  __nv_bfloat16* out;
  int32_t* status;
  const float* bias;
  float scale0, scale1, scale2, shift0, shift1, shift2;
  int T, M, N;
  int kslice_pad;
  int bn, nstage, npass;
  int tmem_cols;
  int num_tiles;
  uint64_t limit_ns;
};

// Shared-memory header (placed before the 1024-aligned tile area).
struct SmemHdr {
  uint64_t a_full[16];
  uint64_t a_empty[16];
  uint64_t b_full[8];
  uint64_t b_empty[8];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  TabHdr tab;
  uint32_t bad[kMaxItems / 32];
  uint32_t still[kMaxItems / 32];
  int start[kMaxItems + 1];
};

__device__ __forceinline__ int tile_kind(int r0, const SmemHdr* h, int T) {
  const int live = h->tab.live;
  if (r0 >= live) return kPad;
  if (T == 1) return kResident;
  const int r1 = min(r0 + kTileM, live) - 1;
  const int n = h->tab.n;
  const int i0 = find_item(h->start, n, r0);
  const int i1 = find_item(h->start, n, r1);
  for (int i = i0; i <= i1; ++i)
    if (!tab_bit(h->still, i) && !tab_bit(h->bad, i)) return kStream;
  return kResident;
}

// Number of K16 MMA steps of block j of a slice (the last block may be partial).
template <int P>
__host__ __device__ constexpr int ksteps_of(int j) {
  constexpr int KS = 3 * P * P;
  const int rem = KS - 64 * j;
  return rem >= 64 ? 4 : (rem + 15) / 16;
}

// One A producer thread writes its row of one temporal slice (all K blocks, in order).
// base: first byte of the patch (top-left pixel, channel 0) in the slice's frame, or
// nullptr for rows written as zeros.  rs: bytes between pixel rows.
template <int P>
__device__ __forceinline__ bool produce_slice(const uint8_t* base, int64_t rs, uint32_t a_smem,
                                              SmemHdr* hs, uint32_t np, int row, const float sc[3],
                                              const float sh[3], volatile int* abort_flag,
                                              uint64_t limit_ns) {
  constexpr int RUN = 3 * P;                 // bytes of one patch row of pixels
  constexpr int KS = 3 * P * P;
  constexpr int NBLK = (KS + 63) / 64;
  constexpr int KEND = ((KS + 15) / 16) * 16;  // features written (K16 padded)
  constexpr int NW = (RUN + 3) / 4 + 1;      // 4-byte words covering a run at any alignment
  constexpr int NA = (RUN + 3) / 4;          // aligned words holding the run
  static_assert(RUN % 2 == 0, "patch rows must hold an even number of bytes");
  const uint32_t empty_parity = (np & 1u) ^ 1u;
  const uint32_t row_off = (uint32_t)row * 128u;
  const uint32_t swz = (uint32_t)(row & 7);
  uint32_t cw[4] = {0u, 0u, 0u, 0u};         // bf16x2 words of the chunk being assembled

  auto emit_word = [&](int kw, uint32_t word) -> bool {
    // kw: index of the bf16 pair inside the slice
    cw[kw & 3] = word;
    if ((kw & 3) == 3) {
      const int kc = kw >> 2;          // chunk of 8 features
      const int j = kc >> 3;           // K block
      const int q = kc & 7;            // chunk inside the 128-byte row
      if (q == 0) {
        if (!mbar_wait(smem_u32(&hs->a_empty[j]), empty_parity, abort_flag, limit_ns)) return false;
      }
      const uint32_t addr = a_smem + (uint32_t)j * kABlockBytes + row_off + (((uint32_t)q ^ swz) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(cw[0]), "r"(cw[1]),
                   "r"(cw[2]), "r"(cw[3])
                   : "memory");
      const bool last_of_block = (q == 7) || (kc == KEND / 8 - 1);
      if (last_of_block) {
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&hs->a_full[j]));
      }
    }
    return true;
  };

#pragma unroll
  for (int ph = 0; ph < P; ++ph) {
    uint32_t al[NA];
    if (base != nullptr) {
      const uint8_t* src = base + (int64_t)ph * rs;
      const uintptr_t a = reinterpret_cast<uintptr_t>(src);
      const uint32_t s = (uint32_t)(a & 3u);
      const uint32_t* w0 = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
      uint32_t raw[NW];
#pragma unroll
      for (int w = 0; w < NW; ++w) raw[w] = (4u * w < s + RUN) ? __ldg(w0 + w) : 0u;
      const uint32_t sel = 0x3210u + 0x1111u * s;
#pragma unroll
      for (int w = 0; w < NA; ++w) al[w] = __byte_perm(raw[w], raw[w + 1], sel);
    } else {
#pragma unroll
      for (int w = 0; w < NA; ++w) al[w] = 0u;
    }
#pragma unroll
    for (int e = 0; e < RUN; e += 2) {
      uint32_t word = 0u;
      if (base != nullptr) {
        const uint32_t src0 = al[e >> 2], src1 = al[(e + 1) >> 2];
        const float v0 = __uint_as_float(__byte_perm(src0, 0x4B000000u, 0x7540u + (e & 3))) - 8388608.0f;
        const float v1 = __uint_as_float(__byte_perm(src1, 0x4B000000u, 0x7540u + ((e + 1) & 3))) - 8388608.0f;
        const float x0 = fmaf(v0, sc[e % 3], sh[e % 3]);
        const float x1 = fmaf(v1, sc[(e + 1) % 3], sh[(e + 1) % 3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(x0, x1);
        word = *reinterpret_cast<uint32_t*>(&p2);
      }
      const int kw = (ph * RUN + e) >> 1;
      if (!emit_word(kw, word)) return false;
    }
  }
  // zero features [KS, KEND) of the last K16 step
#pragma unroll
  for (int k = KS; k < KEND; k += 2)
    if (!emit_word(k >> 1, 0u)) return false;
  (void)NBLK;
  return true;
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1) embed_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                            const EmbedArgs args) {
  constexpr int KS = 3 * P * P;
  constexpr int NBLK = (KS + 63) / 64;
  extern __shared__ uint8_t smem_raw[];
  SmemHdr* hs = reinterpret_cast<SmemHdr*>(smem_raw);
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t tiles_base = (raw_base + (uint32_t)sizeof(SmemHdr) + 1023u) & ~1023u;
  const uint32_t a_smem = tiles_base;
  const uint32_t b_smem = tiles_base + NBLK * kABlockBytes;
  const uint32_t b_stage_bytes = (uint32_t)args.bn * 128u;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &hs->abort_flag;

  // ---- prologue -----------------------------------------------------------
  if (threadIdx.x == 0) {
    hs->abort_flag = 0;
    for (int j = 0; j < NBLK; ++j) {
      mbar_init(smem_u32(&hs->a_full[j]), kProducerThreads);
      mbar_init(smem_u32(&hs->a_empty[j]), 1);
    }
    for (int s = 0; s < args.nstage; ++s) {
      mbar_init(smem_u32(&hs->b_full[s]), 1);
      mbar_init(smem_u32(&hs->b_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&hs->acc_full[b]), 1);
      mbar_init(smem_u32(&hs->acc_empty[b]), kProducerThreads);
    }
    mbar_init(smem_u32(&hs->drain), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    ItemTab tab{hs->start, hs->bad, hs->still, &hs->tab};
    build_item_table(args.items, args.n_items, args.max_items, args.pixel_bytes, P, args.T, args.M,
                     args.rows, 0x7fffffff, tab);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&hs->tmem_base), (uint32_t)args.tmem_cols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) tma_prefetch_desc(&tmap_w);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  write_status(args.status, &hs->tab);
  const uint32_t tmem = hs->tmem_base;

  // ---- roles -------------------------------------------------------------
  if (warp < 4) {
    // A producers
    const float sc[3] = {args.scale0, args.scale1, args.scale2};
    const float sh[3] = {args.shift0, args.shift1, args.shift2};
    const int row = threadIdx.x;
    uint32_t np = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
      const int r0 = tile * kTileM;
      const int kind = tile_kind(r0, hs, args.T);
      if (kind == kPad) continue;
      const int r = r0 + row;
      const uint8_t* base0 = nullptr;
      int64_t rs = 0, fstride = 0;
      if (r < hs->tab.live) {
        const int i = find_item(hs->start, hs->tab.n, r);
        if (!tab_bit(hs->bad, i)) {
          const vitfe_item it = args.items[i];
          int tg, hh, ww;
          decode_local(r - hs->start[i], it.h, it.w, args.M, tg, hh, ww);
          const int64_t H = (int64_t)it.h * P, W = (int64_t)it.w * P;
          rs = W * 3;
          const bool still = (it.frames == 1);
          fstride = still ? 0 : H * W * 3;
          const int64_t f0 = still ? 0 : (int64_t)tg * args.T;
          base0 = args.pixels + it.pixel_offset + ((f0 * H + (int64_t)hh * P) * W + (int64_t)ww * P) * 3;
        }
      }
      const int nprod = (kind == kResident) ? 1 : args.npass * args.T;
      for (int q = 0; ok && q < nprod; ++q) {
        const int s = (kind == kResident) ? 0 : (q % args.T);
        const uint8_t* base = base0 ? base0 + fstride * s : nullptr;
        ok = produce_slice<P>(base, rs, a_smem, hs, np, row, sc, sh, abort_flag, args.limit_ns);
        ++np;
      }
    }
  } else if (warp == kTmaWarp) {
    if (lane == 0) {
      uint32_t nb = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
        const int kind = tile_kind(tile * kTileM, hs, args.T);
        if (kind == kPad) continue;
        for (int p = 0; ok && p < args.npass; ++p) {
          const int n0 = p * args.bn;
          const int nouter = (kind == kResident) ? NBLK : args.T;
          const int ninner = (kind == kResident) ? args.T : NBLK;
          for (int o = 0; ok && o < nouter; ++o) {
            for (int in = 0; ok && in < ninner; ++in) {
              const int j = (kind == kResident) ? o : in;
              const int s = (kind == kResident) ? in : o;
              const uint32_t stage = nb % (uint32_t)args.nstage;
              const uint32_t ph = (nb / (uint32_t)args.nstage) & 1u;
              if (!mbar_wait(smem_u32(&hs->b_empty[stage]), ph ^ 1u, abort_flag, args.limit_ns)) {
                ok = false;
                break;
              }
              const uint32_t full = smem_u32(&hs->b_full[stage]);
              mbar_arrive_expect_tx(full, b_stage_bytes);
              tma_load_2d(b_smem + stage * b_stage_bytes, &tmap_w, full, s * args.kslice_pad + 64 * j, n0);
              ++nb;
            }
          }
        }
      }
      if (!ok) {
        // drain: the last loads of every stage complete on their own
        const uint32_t nlast = nb < (uint32_t)args.nstage ? nb : (uint32_t)args.nstage;
        for (uint32_t d = 1; d <= nlast; ++d) {
          const uint32_t idx = nb - d;
          const uint32_t bar = smem_u32(&hs->b_full[idx % (uint32_t)args.nstage]);
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(bar, (idx / (uint32_t)args.nstage) & 1u) &&
                 global_timer_ns() - t0 < args.limit_ns) {
          }
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      uint32_t nb = 0, na = 0, np = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
        const int kind = tile_kind(tile * kTileM, hs, args.T);
        if (kind == kPad) continue;
        for (int p = 0; ok && p < args.npass; ++p) {
          const uint32_t buf = na & 1u;
          if (!mbar_wait(smem_u32(&hs->acc_empty[buf]), ((na >> 1) & 1u) ^ 1u, abort_flag, args.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int npw = min(args.bn, args.N - p * args.bn);
          const uint32_t idesc = idesc_bf16(kTileM, npw);
          const uint32_t d_tmem = tmem + buf * (uint32_t)args.bn;
          uint32_t accum = 0;
          const int nouter = (kind == kResident) ? NBLK : args.T;
          const int ninner = (kind == kResident) ? args.T : NBLK;
          for (int o = 0; ok && o < nouter; ++o) {
            for (int in = 0; ok && in < ninner; ++in) {
              const int j = (kind == kResident) ? o : in;
              const bool first_use = (kind == kResident) ? (p == 0 && in == 0) : true;
              const bool last_use = (kind == kResident) ? (p == args.npass - 1 && in == ninner - 1) : true;
              if (first_use) {
                if (!mbar_wait(smem_u32(&hs->a_full[j]), np & 1u, abort_flag, args.limit_ns)) {
                  ok = false;
                  break;
                }
              }
              const uint32_t stage = nb % (uint32_t)args.nstage;
              if (!mbar_wait(smem_u32(&hs->b_full[stage]), (nb / (uint32_t)args.nstage) & 1u, abort_flag,
                             args.limit_ns)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_addr = a_smem + (uint32_t)j * kABlockBytes;
              const uint32_t b_addr = b_smem + stage * b_stage_bytes;
              const int nk = ksteps_of<P>(j);
              for (int kk = 0; kk < nk; ++kk) {
                umma_bf16(d_tmem, sw128_desc(a_addr + 32u * kk), sw128_desc(b_addr + 32u * kk), idesc, accum);
                accum = 1;
              }
              umma_commit(smem_u32(&hs->b_empty[stage]));
              ++nb;
              if (last_use) umma_commit(smem_u32(&hs->a_empty[j]));
            }
            if (kind == kStream) ++np;   // one slice production consumed per outer step
          }
          if (!ok) break;
          umma_commit(smem_u32(&hs->acc_full[buf]));
          ++na;
        }
        if (kind == kResident) ++np;
      }
      if (!ok) {
        umma_commit(smem_u32(&hs->drain));
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&hs->drain), 0u) && global_timer_ns() - t0 < args.limit_ns) {
        }
      }
    }
  } else {
    // epilogue warps 4..7: TMEM lanes 32*(warp%4) .. +31
    const int q = warp & 3;
    const int rloc = q * 32 + lane;
    uint32_t na = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
      const int r0 = tile * kTileM;
      const int kind = tile_kind(r0, hs, args.T);
      const int r = r0 + rloc;
      const bool in_bucket = r < args.rows;
      bool valid = false;
      if (r < hs->tab.live) {
        const int i = find_item(hs->start, hs->tab.n, r);
        valid = !tab_bit(hs->bad, i);
      }
      __nv_bfloat16* orow = args.out + (size_t)r * (size_t)args.N;
      if (kind == kPad) {
        if (in_bucket) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          for (int c = 0; c < args.N; c += 8) *reinterpret_cast<uint4*>(orow + c) = z;
        }
        continue;
      }
      for (int p = 0; p < args.npass; ++p) {
        const uint32_t buf = na & 1u;
        if (!mbar_wait(smem_u32(&hs->acc_full[buf]), (na >> 1) & 1u, abort_flag, args.limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int npw = min(args.bn, args.N - p * args.bn);
        for (int c0 = 0; c0 < npw; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + buf * (uint32_t)args.bn + (uint32_t)c0, v);
          tmem_wait_ld();
          if (in_bucket) {
            const int n0 = p * args.bn + c0;
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float y0 = __uint_as_float(v[2 * e]) + __ldg(args.bias + n0 + 2 * e);
              const float y1 = __uint_as_float(v[2 * e + 1]) + __ldg(args.bias + n0 + 2 * e + 1);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(y0, y1);
              pk[e] = valid ? *reinterpret_cast<uint32_t*>(&b2) : 0u;
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + n0);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              __stcs(dst + e, make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]));
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&hs->acc_empty[buf]));
        ++na;
      }
    }
  }

  // ---- teardown ------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, (uint32_t)args.tmem_cols);
  if (threadIdx.x == 0 && hs->abort_flag && args.status != nullptr) {
    args.status[0] = kTimeout;
    args.status[1] = -1;
  }
}

size_t embed_smem_bytes(int nblk, int bn, int nstage) {
  return sizeof(SmemHdr) + 1024 + (size_t)nblk * kABlockBytes + (size_t)nstage * bn * 128;
}

}  // namespace

cudaError_t embed_configure(Ctx& c) {
  c.embed_ok = false;
  // implemented: patch 14 or 16 (Qwen2/2.5-VL and Qwen3-VL); hidden a multiple of 32
  if (!(c.P == 14 || c.P == 16) || (c.N % 32) != 0) return cudaSuccess;
  int max_optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c.device);
  if (e != cudaSuccess) return e;
  const int cand[][2] = {{256, 2}, {128, 3}, {128, 2}};
  for (auto& cb : cand) {
    const int bn = cb[0] > c.N ? c.N : cb[0];
    const size_t need = embed_smem_bytes(c.nblk, bn, cb[1]);
    if (need <= (size_t)max_optin) {
      c.bn = bn;
      c.nstage = cb[1];
      c.embed_smem = need;
      c.embed_ok = true;
      break;
    }
  }
  if (!c.embed_ok) return cudaSuccess;
  if (c.P == 14)
    e = cudaFuncSetAttribute(embed_kernel<14>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.embed_smem);
  else
    e = cudaFuncSetAttribute(embed_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.embed_smem);
  return e;
}

cudaError_t launch_embed(const Ctx& c, const uint8_t* pixels, int64_t pixel_bytes,
                         const vitfe_item* items, const int32_t* n_items, int max_items,
                         int64_t rows, void* out, int32_t* status, cudaStream_t s) {
  EmbedArgs a;
  a.pixels = pixels;
  a.pixel_bytes = pixel_bytes;
  a.items = items;
  a.n_items = n_items;
  a.max_items = max_items;
  a.rows = (int)rows;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.bias = c.bias;
  a.scale0 = c.scale[0]; a.scale1 = c.scale[1]; a.scale2 = c.scale[2];
  a.shift0 = c.shift[0]; a.shift1 = c.shift[1]; a.shift2 = c.shift[2];
  a.T = c.T;
  a.M = c.M;
  a.N = c.N;
  a.kslice_pad = c.kslice_pad;
  a.bn = c.bn;
  a.nstage = c.nstage;
  a.npass = (c.N + c.bn - 1) / c.bn;
  a.tmem_cols = 32;
  while (a.tmem_cols < 2 * c.bn) a.tmem_cols <<= 1;
  a.num_tiles = (int)((rows + kTileM - 1) / kTileM);
  a.limit_ns = c.wait_limit_ns;
  int grid = a.num_tiles < c.sm_count ? a.num_tiles : c.sm_count;
  if (grid < 1) grid = 1;
  if (c.P == 14)
    embed_kernel<14><<<grid, kThreads, c.embed_smem, s>>>(c.tmap_w, a);
  else
    embed_kernel<16><<<grid, kThreads, c.embed_smem, s>>>(c.tmap_w, a);
  return cudaGetLastError();
}

}  // namespace vitfe
