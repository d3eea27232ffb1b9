// Internal definitions shared by the libvitfe translation units (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "vitfe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libvitfe targets Blackwell (build with -gencode arch=compute_103a,code=sm_103a)"
#endif

namespace vitfe {

// ---------------------------------------------------------------------------
// handle
// ---------------------------------------------------------------------------
struct Ctx {
  int device = 0;
  int sm_count = 0;
  // FusedInputNorm folded into one fp32 FMA per value: x = v * scale_c + shift_c,
  // scale_c = rescale / std_c, shift_c = -mean_c / std_c (computed in double, rounded once).
  float scale[3];
  float shift[3];
  int P = 0, T = 0, M = 0, N = 0;
  int kslice = 0;      // 3 * P * P features of one temporal slice, internal order (ph, pw, c)
  int kslice_pad = 0;  // kslice rounded up to 64 (one 128-byte swizzle row of bf16)
  int nblk = 0;        // kslice_pad / 64
  int K = 0;           // 3 * T * P * P (canonical feature width)
  __nv_bfloat16* w_tile = nullptr; // W as the embed kernel's shared-memory images (tile_weight_kernel)
  size_t w_tile_bytes = 0;
  __nv_bfloat16* w_tile_f = nullptr;  // folded-still weight images (one slice: sum of the T slices)
  size_t w_tile_f_bytes = 0;
  float* bias = nullptr;           // [N] fp32 (zeros when no bias)
  static constexpr int kRopeSlots = 4;
  // RoPE axis tables: kRopeSlots cached tables, each keyed by (head_dim, theta) for the
  // handle's lifetime (a slot is never given to another key, so a captured graph that
  // reads a slot stays valid), plus one transient slot rebuilt by every call whose key
  // found no slot.  rope_built[k]: an eager build of slot k has been enqueued.  A build
  // recorded during stream capture runs only when the graph does, so it leaves the slot
  // unbuilt for eager calls.
  float* rope_tab = nullptr;       // (kRopeSlots + 1) x slot_floats
  int rope_hd[kRopeSlots] = {0, 0, 0, 0};
  float rope_theta[kRopeSlots] = {0.f, 0.f, 0.f, 0.f};
  bool rope_built[kRopeSlots] = {false, false, false, false};
  int rope_used = 0;               // slots holding a key
  CUtensorMap tmap_w;              // w_tile viewed as 512-byte rows; a box is one image (bn/8 rows)
  CUtensorMap tmap_wf;             // the same over w_tile_f
  int bn = 0;                      // GEMM N tile of a CTA pair (<= 256)
  int nstage = 0;                  // B pipeline stages
  int max_clusters = 0;            // co-resident CTA pairs of the embed kernel
  size_t embed_smem = 0;           // dynamic shared memory of the embed kernel
  bool embed_ok = false;           // embed kernel supports this shape
  uint64_t wait_limit_ns = 1000000000ull;
  // failure-detection test hook (VITFE_TEST_STALL_W_LOADS=1 at create): the embed kernel's
  // weight producer issues no loads, so the MMA's bounded wait runs out and the launch
  // reports VITFE_EDEVICE_TIMEOUT
  bool test_stall_w_loads = false;
  int np_per_sm = 1;               // resident CTAs per SM of the specialised normalise+patchify kernel
  // host-buffer pipeline of vitfe_embed_rope_host: created on first use, grown on demand
  struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t up[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr}, down[2] = {nullptr, nullptr};
    uint8_t* px[2] = {nullptr, nullptr};
    size_t px_cap = 0;
    vitfe_item* items[2] = {nullptr, nullptr};   // VITFE_MAX_ITEMS each
    int32_t* n[2] = {nullptr, nullptr};
    int32_t* status[2] = {nullptr, nullptr};
    __nv_bfloat16* out[2] = {nullptr, nullptr};
    float* cos[2] = {nullptr, nullptr};
    float* sin[2] = {nullptr, nullptr};
    int64_t rows_cap = 0;
    int hd_cap = 0;
    // page-locked host staging of the per-run descriptors, counts and status words: a copy
    // from or to pageable memory would block the host and serialise the pipeline
    vitfe_item* h_items = nullptr;
    int32_t* h_small = nullptr;     // [runs] counts, then [runs][2] status words
    size_t h_items_cap = 0, h_small_cap = 0;
  } pipe;
};

constexpr int kMaxItems = VITFE_MAX_ITEMS;
constexpr int kTileM = 128;

// status codes written on the device
enum : int { kOk = 0, kDesc = VITFE_EDEVICE_DESC, kRange = VITFE_EDEVICE_RANGE,
             kTimeout = VITFE_EDEVICE_TIMEOUT };

// ---------------------------------------------------------------------------
// item table (built by every kernel's CTA into shared memory)
// ---------------------------------------------------------------------------
struct TabHdr {
  int n;          // items considered
  int live;       // live rows inside the bucket (min(sum rows, bucket))
  int code;       // first device error
  int bad_item;   // its item index (-1: none / whole call)
  int maxside;    // max(h, w) over valid items
};

struct ItemTab {
  int* start;       // [n + 1] clamped to the bucket
  uint32_t* bad;    // bit i: item i is invalid (rows written as pad)
  uint32_t* still;  // bit i: item i is a still (one stored frame)
  TabHdr* hdr;
};

__device__ __forceinline__ bool tab_bit(const uint32_t* m, int i) { return (m[i >> 5] >> (i & 31)) & 1u; }

// Built by warp 0 of the calling CTA; the caller synchronises the CTA afterwards.
// pixel_bytes < 0 skips the pixel-range checks (kernels that read no pixels).
__device__ inline void build_item_table(const vitfe_item* __restrict__ items,
                                        const int32_t* __restrict__ n_items, int max_items,
                                        int64_t pixel_bytes, int P, int T, int M, int64_t bucket,
                                        int max_side_limit, ItemTab tab) {
  const int lane = threadIdx.x & 31;
  int n = __ldg(n_items);
  int code = kOk, bad_item = -1;
  if (n < 0 || n > max_items) { code = kDesc; n = 0; }
  long long carry = 0;
  int maxside = 0;
  int first_over = -1;   // first item that does not fit entirely inside the bucket
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    long long r = 0;
    int ecode = kOk;
    bool still = false;
    if (i < n) {
      const vitfe_item it = items[i];
      const long long t = it.t, h = it.h, w = it.w;
      if (t < 0 || h < 0 || w < 0 || t * h * w > 0x7fffffffLL) {
        ecode = kDesc;
      } else {
        r = t * h * w;
        still = (it.frames == 1);
        if ((h % M) || (w % M)) ecode = kDesc;
        else if (still ? (t != 1) : ((long long)it.frames != t * T)) ecode = kDesc;
        else if (h > max_side_limit || w > max_side_limit) ecode = kDesc;
        else if (pixel_bytes >= 0) {
          const long long frames = it.frames;
          const long long bytes = frames * (h * P) * (w * P) * 3;
          if (it.pixel_offset < 0 || (it.pixel_offset & 15)) ecode = kDesc;
          else if (it.pixel_offset + bytes > pixel_bytes) ecode = kRange;
        }
        if (ecode == kOk) maxside = max(maxside, (int)max(h, w));
      }
    }
    // inclusive scan of r across the warp
    long long incl = r;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      long long o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    const long long excl = carry + incl - r;
    if (i < n) tab.start[i] = (int)min(excl, (long long)bucket);
    const uint32_t overm = __ballot_sync(0xffffffffu, i < n && excl + r > bucket);
    if (first_over < 0 && overm) first_over = base + __ffs(overm) - 1;
    const uint32_t badm = __ballot_sync(0xffffffffu, ecode != kOk);
    const uint32_t stillm = __ballot_sync(0xffffffffu, still);
    if (lane == 0) { tab.bad[base >> 5] = badm; tab.still[base >> 5] = stillm; }
    if (code == kOk && badm) {
      const int src = __ffs(badm) - 1;
      code = __shfl_sync(0xffffffffu, ecode, src);
      bad_item = base + src;
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) maxside = max(maxside, __shfl_xor_sync(0xffffffffu, maxside, d));
  if (lane == 0) {
    tab.start[n] = (int)min(carry, (long long)bucket);
    if (carry > bucket && code == kOk) {
      code = kRange;
      bad_item = first_over;
    }
    tab.hdr->n = n;
    tab.hdr->live = (int)min(carry, (long long)bucket);
    tab.hdr->code = code;
    tab.hdr->bad_item = bad_item;
    tab.hdr->maxside = maxside;
  }
}

// Largest i in [0, n) with start[i] <= r (requires r < start[n]).
__device__ __forceinline__ int find_item(const int* start, int n, int r) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

struct RowPos {
  int item;
  int tg, hh, ww;   // temporal group, patch row, patch column
};

// Merge-order decode of a row local to its item ("vLLM 多模态推理｜ViT 性能优化", §2.2
// step (1) and §3.3 step 2): local = ((tg*(h/m) + hb)*(w/m) + wb)*m*m + mh*m + mw.
__device__ __forceinline__ void decode_local(int local, int h, int w, int M, int& tg, int& hh, int& ww) {
  const int hw = h * w;
  tg = local / hw;
  const int rem = local - tg * hw;
  const int mm = M * M;
  const int g = rem / mm;
  const int within = rem - g * mm;
  const int uw = w / M;
  const int hb = g / uw;
  const int wb = g - hb * uw;
  const int mh = within / M;
  const int mw = within - mh * M;
  hh = hb * M + mh;
  ww = wb * M + mw;
}

// Programmatic dependent launch.  grid_dep_trigger: this CTA lets the next kernel of the
// stream (launched with programmatic stream serialization) begin once every CTA of this grid
// has triggered or exited.  grid_dep_wait: block until the previous kernel of the stream has
// completed and its memory is visible (returns at once when there is none to wait for).
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Only CTA 0 writes the status pair; a timeout anywhere overrides it later.
__device__ __forceinline__ void write_status(int32_t* status, const TabHdr* hdr) {
  if (status != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    status[0] = hdr->code;
    status[1] = hdr->bad_item;
  }
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase of `parity` has completed; false when the
// CTA-wide abort flag is set or the wait exceeded `limit_ns` (then it sets the flag).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// TMA: 2-D tiled load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// tcgen05 (5th-generation tensor core, accumulators in tensor memory)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D(tmem) (+)= A(smem) * B(smem)^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when all tcgen05 ops issued so far by this thread complete.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base lane + i), cols [c, c+32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Weight images per (N pass, CTA half) for TL temporal slices of kslice features: one per
// (slice, 64-feature block), except that when the last block of a slice holds at most 16
// features (one K16 step) the TL slices' tails share one image, slice s at K16 offset s.
__host__ __device__ constexpr bool w_tail_shared(int kslice) {
  return (kslice % 64) != 0 && (kslice % 64) <= 16;
}
__host__ __device__ constexpr int w_images(int kslice, int TL) {
  return w_tail_shared(kslice) ? TL * (kslice / 64) + 1 : TL * ((kslice + 63) / 64);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row core groups 1024 bytes apart (tile base 1024-byte aligned).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);        // start address
  d |= (uint64_t)1u << 16;                          // leading byte offset (unused with swizzle)
  d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset: 8 rows * 128 B
  d |= (uint64_t)1u << 46;                          // descriptor version (tcgen05)
  d |= (uint64_t)2u << 61;                          // swizzle: 128-byte
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (K-major), fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                       // D format: f32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// ---------------------------------------------------------------------------
// CTA-pair (cluster of 2) variants: one MMA spans the two CTAs' shared memory and
// tensor memory; barriers of the even (leader) CTA are reached through the cluster
// shared window.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// A relaxed remote arrive: a completion signal only, ordering nothing.  Used where an
// earlier release (to a barrier the waiter acquires first) already made the data visible.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (barriers that peers arrive on).  Waiters off
// the MMA-issue path pass sleep_ns > 0: after a few failed polls they back off with
// __nanosleep so that they do not take issue slots from the warps that feed the tensor core.
// The first poll is inline; the polling loop is one out-of-line copy (the waits sit in fully
// unrolled loops, and inline copies of the loop would multiply the code the SM fetches).
static __device__ __noinline__ bool mbar_wait_cl_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               uint64_t limit_ns, uint32_t sleep_ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (sleep_ns && i > 2) __nanosleep(sleep_ns);
    if ((i & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t limit_ns, uint32_t sleep_ns = 0) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return mbar_wait_cl_slow(bar, parity, abort_flag, limit_ns, sleep_ns);
}
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}
// TMA load into this CTA's shared memory, completion counted on a barrier that may live
// in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (both CTAs' tensor memory, 128 lanes each) (+)= A (both CTAs' smem, 128 rows each)
// * B^T (N/2 rows in each CTA's smem); issued by one thread of the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with A in tensor memory: each CTA's 128 lanes hold its 128 rows of A, column c
// the bf16 pair of features (2c, 2c+1); one K16 step spans 8 columns from a_tmem.
__device__ __forceinline__ void umma_bf16_pair_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 4 consecutive 32-bit columns from registers (warp-collective; warp w of a
// CTA reaches lanes [32 (w % 4), 32 (w % 4) + 32)).
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// One lane of a converged warp is elected (the same lane every time for a full warp).
__device__ __forceinline__ bool elect_one() {
  uint32_t p = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(p));
  return p != 0;
}

// Bounded mbarrier wait by a whole converged warp (acquire at CTA or cluster scope).  The
// lanes vote on every poll, so they all return together and with the same value: true when
// the phase of `parity` has completed, false (and *abort_flag set) when the abort flag was
// raised or `limit_ns` passed first.
template <bool kCluster>
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
  if constexpr (kCluster) return mbar_try_wait_cluster(bar, parity);
  else return mbar_try_wait(bar, parity);
}
// sleep_ns > 0: after a few failed polls the warp backs off with __nanosleep, leaving its
// scheduler's issue slots to the warps it shares them with.  As for mbar_wait_cl, the first
// poll is inline and the loop out of line.
template <bool kCluster>
static __device__ __noinline__ bool mbar_wait_warp_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                 uint64_t limit_ns, uint32_t sleep_ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (__all_sync(0xffffffffu, mbar_poll<kCluster>(bar, parity))) return true;
    if (sleep_ns && i > 2) __nanosleep(sleep_ns);
    if ((i & 15u) == 0) {
      const bool stop = *abort_flag != 0 || global_timer_ns() - t0 > limit_ns;
      if (__any_sync(0xffffffffu, stop)) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}
template <bool kCluster>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               uint64_t limit_ns, uint32_t sleep_ns = 0) {
  if (__all_sync(0xffffffffu, mbar_poll<kCluster>(bar, parity))) return true;
  return mbar_wait_warp_slow<kCluster>(bar, parity, abort_flag, limit_ns, sleep_ns);
}

// Arrive once on the barrier at offset `bar` in both CTAs of the pair when all prior
// tcgen05 ops of this thread complete.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(mask)
      : "memory");
}

// ---------------------------------------------------------------------------
// launchers (defined in the kernel translation units)
// ---------------------------------------------------------------------------
// rope_cos != nullptr: the same launch also writes the 2D-RoPE rows from rope_tab
// (an axis table from rope_table_for; nf = head_dim / 4).
// folded: still tiles use the folded-still weight (one slice of K).
cudaError_t launch_embed(const Ctx& c, const uint8_t* pixels, int64_t pixel_bytes,
                         const vitfe_item* items, const int32_t* n_items, int max_items,
                         int64_t rows, void* out, int32_t* status, cudaStream_t s,
                         const float* rope_tab = nullptr, int rope_nf = 0, float* rope_cos = nullptr,
                         float* rope_sin = nullptr, bool folded = false);
cudaError_t embed_configure(Ctx& c);
cudaError_t np_configure(Ctx& c);   // at create: the normalise+patchify kernel's smem and occupancy
// The handle's cos/sin axis table of (head_dim, theta): found in its slots, or built there
// (one launch on `s`) the first time.  Layout: cos at [p * nf + i], sin at
// [VITFE_ROPE_MAX_SIDE * nf + p * nf + i], nf = head_dim / 4, p < VITFE_ROPE_MAX_SIDE.
cudaError_t rope_table_for(Ctx& c, int head_dim, float theta, cudaStream_t s, const float** tab_out);
cudaError_t launch_rope(Ctx& c, const vitfe_item* items, const int32_t* n_items,
                        int max_items, int64_t rows, int head_dim, float theta, float* cos,
                        float* sin, int32_t* status, cudaStream_t s);
cudaError_t launch_normalize_patchify(const Ctx& c, const uint8_t* pixels, int64_t pixel_bytes,
                                      const vitfe_item* items, const int32_t* n_items,
                                      int max_items, int64_t rows, void* out, int32_t* status,
                                      cudaStream_t s);
cudaError_t launch_rope_apply(const float* cos, const float* sin, int64_t rows, int head_dim, void* q,
                              int heads_q, int64_t q_stride, void* k, int heads_k, int64_t k_stride,
                              cudaStream_t s);
cudaError_t launch_cu_seqlens(const Ctx& c, const vitfe_item* items, const int32_t* n_items, int max_items,
                              int64_t rows, int max_seqs, int32_t* cu, int32_t* info, int32_t* status,
                              cudaStream_t s);
cudaError_t launch_pos_ids(const Ctx& c, const vitfe_item* items, const int32_t* n_items,
                           int max_items, int64_t rows, int32_t* pos, int32_t* status,
                           cudaStream_t s);
cudaError_t launch_tile_weight(const Ctx& c, const __nv_bfloat16* W, const __nv_bfloat16* b,
                                  cudaStream_t s);

}  // namespace vitfe
