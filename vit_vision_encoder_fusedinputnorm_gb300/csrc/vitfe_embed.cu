// Fused FusedInputNorm + merge-order patchify + patch-embed GEMM + bias (sm_103a).
//
// What it computes ("PR #55370 完整报告" 实现拆解 item 2; "vLLM 多模态推理｜ViT 性能优化"
// §2.2 and §3.2): for every patch row r (items in order, merge order inside an item)
//     out[r][n] = bf16( sum_k A[r][k] * W[n][k] + b[n] ),
//     A[r][k]   = bf16( v * rescale/std_c - mean_c/std_c ),
// where v is the uint8 pixel feature k of patch r.  A never reaches device memory.
//
// Structure: persistent clusters of two CTAs (one per SM).  A pair owns 256-row tiles,
// 128 rows per CTA; one tcgen05.mma.cta_group::2 (M=256) spans both CTAs' shared and
// tensor memory, so each CTA holds only half of every W tile.  Per CTA, 16 warps (their
// numbers, chosen per sub-partition, are listed with the role helpers below):
//   8 warps     A producers: two threads per tile row (each half of the K blocks) gather
//               uint8 pixel runs with aligned 4-byte loads, normalise in fp32, round to
//               bf16 and store into 128-byte-swizzled K-major shared-memory blocks (64
//               features each); with patch 16 the last two blocks of each half go to
//               tensor memory instead (tcgen05.st), and the MMA reads them from there;
//   2 warps     TMA producers of this CTA's half of each W tile, alternate stages: one
//               box copies one shared-memory image of the pre-tiled weight (bn/8 rows of
//               512 bytes);
//   MMA warp    tensor-memory allocation (both CTAs); in the even CTA the whole warp runs
//               the MMA issue loop and one elected lane issues (fp32 accumulators
//               double-buffered in tensor memory; N passes of 256 columns, or 192 with
//               patch 16 so that the A blocks fit beside them);
//   4 warps     epilogue, one warp per tensor-memory lane quarter: tcgen05.ld of the
//               accumulator, + bias, bf16 RNE, 256-bit stores; in a vitfe_embed_rope
//               launch also the tile's 2D-RoPE rows.
// Barriers that gather both CTAs (A ready, W tile ready, accumulator free) live in the
// even CTA; the MMA's completion is multicast to both CTAs.
//
// Features inside one temporal slice are ordered (ph, pw, c) so that each patch row
// of pixels is one contiguous byte run; the weight was permuted the same way once
// at create.  The whole slice of A (all K blocks) stays resident in shared memory
// while the tile loops over the N passes; for stills the temporal slices are equal,
// so one resident slice feeds the MMAs of every slice ("resident" tiles).  Tiles
// holding video rows re-produce A per slice ("stream" tiles), once for each pair of N
// passes: every A block then feeds both tensor-memory accumulators before it is freed.
//
// The K blocks are consumed in the order the producer threads fill them (one block of each
// producer range in turn).  The work unit is (pair tile, group of N passes): the tiles of
// a last round with fewer tiles than CTA pairs have their passes spread over several pairs.
//
// Every mbarrier wait is bounded (global timer); on expiry the CTA drains its async
// copies and MMAs, frees its tensor memory, writes VITFE_EDEVICE_TIMEOUT and exits.
#include "vitfe_internal.cuh"

namespace vitfe {
namespace {

constexpr int kThreads = 512;            // 16 warps
constexpr int kProducerThreads = 128;     // tile rows of a CTA (two producer threads each)
constexpr int kEpilogueThreads = 128;     // one warp per tensor-memory lane quarter
constexpr int kPairRows = 2 * kTileM;
// Weight stages are loaded by two warps in turn.  With one loading warp the ring delivered
// about 22 bytes per clock into each SM whatever its depth, below the 32 bytes per clock the
// MMA consumes; two warps deliver the full rate.
constexpr int kWLoaders = 2;
constexpr int kABlockBytes = kTileM * 128;   // 128 rows x 64 bf16

// Warp roles.  Warp w issues on SM sub-partition w % 4.  The producers' conversion is dense
// ALU work, and a sub-partition shared with it slows the MMA issue loop and the weight loads;
// so with patch 14 the MMA warp sits on sub-partition 3 with one weight-loading warp and its
// epilogue warp only, the eight producer warps on 0-2, the other loader on 2:
//   producers 0, 1, 2, 4 (half 0) and 5, 6, 8, 9 (half 1); MMA 3; weight loads 7, 10;
//   epilogue 12-15 (lane quarter w % 4); A-block forwarder 11 (odd CTA; idle in the even).
// Patch 16's producers also write tensor memory, where warp w reaches only lane quarter
// w % 4, so their eight warps must cover every quarter twice: producers 0-7, epilogue 8-11,
// weight loads 12 and 14, MMA 13, A-block forwarder 15.
// A cluster-scope release costs about 1.4 k cycles, which producer warps arriving on the
// even CTA's barrier would pay on every block.  So the even CTA's producers arrive with
// CTA scope on its a_full barriers directly, and the odd CTA's arrive with CTA scope on
// their own a_local barriers; the odd CTA's forwarder passes those on to the even CTA two
// blocks at a time, in the MMA's consumption order: one release, which the MMA acquires
// with the first of the two blocks, then a relaxed arrival for the second.
template <int P>
__host__ __device__ constexpr bool split_roles() { return P != 16; }   // patch 16: A blocks in tensor memory
template <int P>
__device__ __forceinline__ int producer_index(int w) {   // 0..7, or -1 for other roles
  if (!split_roles<P>()) return w < 8 ? w : -1;
  return w < 3 ? w : (w == 4 ? 3 : (w == 5 || w == 6) ? w - 1 : (w == 8 || w == 9) ? w - 2 : -1);
}
template <int P>
__host__ __device__ constexpr int mma_warp() { return split_roles<P>() ? 3 : 13; }
template <int P>
__host__ __device__ constexpr int w_load_warp(int i) { return split_roles<P>() ? (i ? 10 : 7) : 12 + 2 * i; }
template <int P>
__host__ __device__ constexpr bool epilogue_warp(int w) { return split_roles<P>() ? w >= 12 : (w >= 8 && w < 12); }
template <int P>
__host__ __device__ constexpr int forward_warp() { return split_roles<P>() ? 11 : 15; }

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
  int bn, nstage, npass;
  int tmem_cols;
  int num_tiles;   // 256-row pair tiles
  // work units: tiles [0, whole_tiles) are one unit each (all npass N passes); every later
  // tile is `split` units of ppu passes each (unit whole_tiles + (tile - whole_tiles) *
  // split + group), so that a last round holding fewer tiles than CTA pairs is spread
  // over the pairs
  int whole_tiles, split, ppu, num_units;
  uint64_t limit_ns;
  int stall_w_loads;       // test hook: the weight producer issues nothing
  // 2D-RoPE rows written by the same launch (null: embeddings only)
  const float* rope_tab;   // the handle's axis table: cos [p * nf + i], sin after VITFE_ROPE_MAX_SIDE rows
  float* rope_cos;
  float* rope_sin;
  int rope_nf;             // head_dim / 4
  int folded;              // still tiles multiply one slice of A by the folded-still weight
};

// Shared-memory header (placed before the 1024-aligned tile area).
struct SmemHdr {
  uint64_t a_full[16];     // even CTA: block j of both CTAs is ready (its own producer warps
                           // and one forward from the odd CTA)
  uint64_t a_local[16];    // odd CTA: this CTA's producer warps have written block j
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
  const int r1 = min(r0 + kPairRows, live) - 1;
  const int n = h->tab.n;
  const int i0 = find_item(h->start, n, r0);
  const int i1 = find_item(h->start, n, r1);
  for (int i = i0; i <= i1; ++i)
    if (!tab_bit(h->still, i) && !tab_bit(h->bad, i)) return kStream;
  return kResident;
}

// Tile and N-pass range [p_lo, p_hi) of work unit u.
__device__ __forceinline__ void unit_range(const EmbedArgs& a, int u, int& tile, int& p_lo, int& p_hi) {
  if (u < a.whole_tiles) {
    tile = u;
    p_lo = 0;
    p_hi = a.npass;
    return;
  }
  const int v = u - a.whole_tiles;
  const int g = v % a.split;
  tile = a.whole_tiles + v / a.split;
  p_lo = g * a.ppu;
  p_hi = min(a.npass, p_lo + a.ppu);
}

// Number of K16 MMA steps of block j of a slice (the last block may be partial).
template <int P>
__host__ __device__ constexpr int ksteps_of(int j) {
  constexpr int KS = 3 * P * P;
  const int rem = KS - 64 * j;
  return rem >= 64 ? 4 : (rem + 15) / 16;
}

// Where the K blocks of A live.  Patch 16 keeps the last two blocks of each producer half
// in tensor memory, beside accumulators of at most 192 columns each: the 64 KB that frees
// in shared memory holds six more W stages.  Patch 14 keeps every block in shared memory.
constexpr uint32_t kTmemACol = 384;   // first tensor-memory column of the A blocks
template <int P>
__host__ __device__ constexpr int ntm_blocks() { return P == 16 ? 4 : 0; }
template <int P>
__host__ __device__ constexpr int nblk_of() { return (3 * P * P + 63) / 64; }
template <int P>
__host__ __device__ constexpr bool in_tmem(int j) {
  constexpr int H = nblk_of<P>() / 2, Q = ntm_blocks<P>() / 2;
  return Q > 0 && (j % H) >= H - Q;
}
// tensor-memory column of block j (in_tmem), 32 columns per block
template <int P>
__host__ __device__ constexpr uint32_t tm_col(int j) {
  constexpr int H = nblk_of<P>() / 2, Q = ntm_blocks<P>() / 2;
  return kTmemACol + 32u * (uint32_t)((j / H) * Q + (j % H) - (H - Q));
}
// shared-memory slot of block j (!in_tmem)
template <int P>
__host__ __device__ constexpr int smem_slot(int j) {
  constexpr int H = nblk_of<P>() / 2, Q = ntm_blocks<P>() / 2;
  return (j / H) * (H - Q) + (j % H);
}

// Order in which the MMA consumes (and, in a tile's last pass, releases) the K blocks of
// a slice: 0, NBLK/2, 1, NBLK/2 + 1, ...  The two producer threads of a row fill blocks
// [0, NBLK/2) and [NBLK/2, NBLK) in parallel, so this order consumes both halves at the
// pace they are filled, and frees both early for the next tile.
template <int NBLK>
__host__ __device__ constexpr int blk_order(int jj) {
  static_assert(NBLK % 2 == 0, "two producer halves of equal size");
  return (jj & 1) ? NBLK / 2 + jj / 2 : jj / 2;
}

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

// One A producer thread writes K blocks [JB, JE) of its row of one temporal slice, in
// order.  base: first byte of the patch (top-left pixel, channel 0) in the slice's frame,
// or nullptr for rows written as zeros.  rs: bytes between pixel rows.  Two threads share
// a row (one per half of the K blocks), so that two producer warps per SM sub-partition
// hide each other's load latency.
//
// Schedule per K block j: convert and store its 64 features, make them visible to the
// tensor core (proxy fence + CTA-scope release arrive on this CTA's a_local barrier, which
// the forwarder warp passes on), then wait for block j+1's shared-memory slot to be freed.
// The pixel rows are loaded two rows ahead (row r+2 as soon as row r has been realigned),
// so a row's load latency overlaps the conversion of the row before it; a load may then
// still be in flight at a release arrive, which waits for it, but it was issued a row's
// conversion earlier (before, the loads of block j+1 were issued after block j's arrive and
// their whole latency came before block j+1's conversion).
template <int P, int JB, int JE>
__device__ __forceinline__ bool produce_blocks(const uint8_t* base, int64_t rs, uint32_t a_smem,
                                               SmemHdr* hs, uint32_t np, int row, const float sc[3],
                                               const float sh[3], volatile int* abort_flag,
                                               uint64_t limit_ns, uint32_t a_local0, uint32_t tmem_a) {
  constexpr int RUN = 3 * P;                 // bytes of one patch row of pixels
  constexpr int KS = 3 * P * P;
  constexpr int NBLK = (KS + 63) / 64;
  constexpr int KEND = ((KS + 15) / 16) * 16;  // features written (K16 padded)
  constexpr int NW = (RUN + 3) / 4 + 1;      // 4-byte words covering a run at any alignment
  constexpr int NA = (RUN + 3) / 4;          // aligned words holding the run
  constexpr int E0 = 64 * JB;                // first feature of the range
  constexpr int E1 = (64 * JE < KEND) ? 64 * JE : KEND;   // one past the last feature written
  constexpr int R0 = E0 / RUN;               // first pixel row touched
  constexpr int RL = ((E1 < KS ? E1 : KS) - 1) / RUN;      // last pixel row touched
  // Register ring of loaded pixel rows: row r+2 goes into row r's slot right after row r
  // has been realigned into al[], so two slots suffice.
  constexpr int R = 2;
  static_assert(RUN % 2 == 0 && RUN > 32, "patch rows: even length, at most two start per block");
  static_assert(NBLK <= 16 && JB < JE && JE <= NBLK, "A slots");
  // (scale, shift) of the channel pairs (c, c+1 mod 3) that a feature pair starting at
  // channel c covers
  const uint64_t sc2[3] = {pack2(__float_as_uint(sc[0]), __float_as_uint(sc[1])),
                           pack2(__float_as_uint(sc[1]), __float_as_uint(sc[2])),
                           pack2(__float_as_uint(sc[2]), __float_as_uint(sc[0]))};
  const uint64_t sh2[3] = {pack2(__float_as_uint(sh[0]), __float_as_uint(sh[1])),
                           pack2(__float_as_uint(sh[1]), __float_as_uint(sh[2])),
                           pack2(__float_as_uint(sh[2]), __float_as_uint(sh[0]))};
  const uint32_t empty_parity = (np & 1u) ^ 1u;
  const uint32_t row_off = (uint32_t)row * 128u;
  const uint32_t swz = (uint32_t)(row & 7);
  uint32_t cw[4] = {0u, 0u, 0u, 0u};         // bf16x2 words of the chunk being assembled
  uint32_t raw[R][NW];
  const uint32_t a_empty0 = smem_u32(&hs->a_empty[0]);

#define VITFE_LOAD_ROW(PH)                                                                  \
  do {                                                                                       \
    if (base != nullptr) {                                                                   \
      const uintptr_t a_ = reinterpret_cast<uintptr_t>(base + (int64_t)(PH) * rs);          \
      const uint32_t s_ = (uint32_t)(a_ & 3u);                                               \
      const uint32_t* w0_ = reinterpret_cast<const uint32_t*>(a_ & ~uintptr_t(3));           \
      _Pragma("unroll") for (int w_ = 0; w_ < NW; ++w_)                                     \
        raw[(PH) % R][w_] = (4u * w_ < s_ + RUN) ? __ldg(w0_ + w_) : 0u;                     \
    }                                                                                        \
  } while (0)
  // the range's first two rows (the first may have started in an earlier block), then the
  // first block's slot; every later row is loaded two rows ahead, as soon as the row that
  // held its register slot has been realigned, so that its latency overlaps the conversion
  // of the row in between
  VITFE_LOAD_ROW(R0);
  if (R0 + 1 <= RL && R0 + 1 < P) VITFE_LOAD_ROW(R0 + 1);
  if (!mbar_wait_cl(a_empty0 + 8u * JB, empty_parity, abort_flag, limit_ns)) return false;
  if (in_tmem<P>(JB)) tc_fence_after();

#pragma unroll
  for (int ph = R0; ph <= P; ++ph) {
    // ph == P: the zero features [KS, KEND) of the last K16 step
    if (ph > RL && ph < P) continue;
    if (ph == P && E1 <= KS) continue;
    uint32_t al[NA];
    if (ph < P && base != nullptr) {
      const uint32_t sl = 0x3210u + 0x1111u * (uint32_t)(reinterpret_cast<uintptr_t>(base + (int64_t)ph * rs) & 3u);
#pragma unroll
      for (int w = 0; w < NA; ++w) al[w] = __byte_perm(raw[ph % R][w], raw[ph % R][w + 1], sl);
      if (ph + 2 <= RL && ph + 2 < P) VITFE_LOAD_ROW(ph + 2);
    } else {
#pragma unroll
      for (int w = 0; w < NA; ++w) al[w] = 0u;
    }
    const int row_start = (ph < P) ? ph * RUN : KS;
    const int row_end = (ph < P) ? (ph + 1) * RUN : KEND;
    const int e_lo = (row_start < E0 ? E0 : row_start) - row_start;
    const int e_hi = (row_end > E1 ? E1 : row_end) - row_start;
#pragma unroll
    for (int e = 0; e < RUN; e += 2) {
      if (e < e_lo || e >= e_hi) continue;
      uint32_t word = 0u;
      if (ph < P && base != nullptr) {
        const uint32_t b0 = __byte_perm(al[e >> 2], 0x4B000000u, 0x7540u + (e & 3));
        const uint32_t b1 = __byte_perm(al[(e + 1) >> 2], 0x4B000000u, 0x7540u + ((e + 1) & 3));
        uint32_t x0, x1;
        unpack2(norm2(pack2(b0, b1), sc2[e % 3], sh2[e % 3]), x0, x1);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(x0), __uint_as_float(x1));
        word = *reinterpret_cast<uint32_t*>(&p2);
      }
      const int kw = (row_start + e) >> 1;     // bf16 pair inside the slice
      cw[kw & 3] = word;
      if ((kw & 3) == 3) {
        const int kc = kw >> 2;                // chunk of 8 features
        const int j = kc >> 3;                 // K block
        const int q = kc & 7;                  // chunk inside the 128-byte row
        if (in_tmem<P>(j)) {
          // four columns of this thread's tensor-memory lane (warp-collective)
          tmem_st_32x32b_x4(tmem_a + tm_col<P>(j) + 4u * (uint32_t)q, cw[0], cw[1], cw[2], cw[3]);
        } else {
          const uint32_t addr =
              a_smem + (uint32_t)smem_slot<P>(j) * kABlockBytes + row_off + (((uint32_t)q ^ swz) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(cw[0]), "r"(cw[1]), "r"(cw[2]),
                       "r"(cw[3])
                       : "memory");
        }
        if (q == 7 || kc == KEND / 8 - 1) {
          // this thread's writes become visible to the tensor core (generic-proxy shared
          // memory: proxy fence; tensor memory: wait for the stores, then the tcgen05
          // fence); one CTA-scope release arrive per warp: on a_full in the even CTA, on
          // a_local in the odd one (passed on by its forwarder)
          if (in_tmem<P>(j)) {
            tmem_wait_st();
            tc_fence_before();
          } else {
            fence_proxy_async_smem();
          }
          __syncwarp();
          if ((threadIdx.x & 31) == 0) mbar_arrive(a_local0 + 8u * (uint32_t)j);
          if (j + 1 < JE) {
            if (!mbar_wait_cl(a_empty0 + 8u * (uint32_t)(j + 1), empty_parity, abort_flag, limit_ns))
              return false;
            if (in_tmem<P>(j + 1)) tc_fence_after();
          }
        }
      }
    }
  }
#undef VITFE_LOAD_ROW
  return true;
}

// 2D-RoPE rows ("vLLM 多模态推理｜ViT 性能优化" §3.3 step 3) of 32 consecutive rows
// [wbase, wbase + 32), one per lane (hp, wp: the lane's row position, -1 for pad rows and
// rows of invalid items): cos[r] = [tab_cos[hp][0..nf) || tab_cos[wp][0..nf)], sin
// likewise, pad rows (1, 0).  The warp writes the rows' contiguous range with float4
// stores; every lane of the warp calls it.
__device__ __forceinline__ void rope_rows(const EmbedArgs& a, int wbase, int hp, int wp, int lane) {
  constexpr int kBatch = 4;          // float4 groups per lane whose table loads are in flight together
  const int nf = a.rope_nf;
  const int width = 2 * nf;          // floats per row
  const int nvec = width >> 2;       // float4 per row (head_dim % 8 == 0)
  const int cnt = min(32, a.rows - wbase);
  if (cnt <= 0) return;
  const int total = cnt * nvec;
  const float* __restrict__ tc = a.rope_tab;
  const float* __restrict__ ts = a.rope_tab + (size_t)VITFE_ROPE_MAX_SIDE * nf;
  const bool vec_tab = (nf % 4) == 0;
  float4* cdst = reinterpret_cast<float4*>(a.rope_cos + (size_t)wbase * width);
  float4* sdst = reinterpret_cast<float4*>(a.rope_sin + (size_t)wbase * width);
  for (int f0 = 0; f0 < total; f0 += 32 * kBatch) {
    float4 cv[kBatch], sv[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int f = f0 + 32 * k + lane;
      const int rr = min(f / nvec, 31);
      const int h = __shfl_sync(0xffffffffu, hp, rr);
      const int w = __shfl_sync(0xffffffffu, wp, rr);
      cv[k] = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
      sv[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (f < total && h >= 0) {
        const int col = 4 * (f - rr * nvec);
        if (vec_tab) {
          const int p = col < nf ? h : w;
          const int i = col < nf ? col : col - nf;
          cv[k] = __ldg(reinterpret_cast<const float4*>(tc + (size_t)p * nf + i));
          sv[k] = __ldg(reinterpret_cast<const float4*>(ts + (size_t)p * nf + i));
        } else {
          float c4[4], s4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cc = col + e;
            const int p = cc < nf ? h : w;
            const int i = cc < nf ? cc : cc - nf;
            c4[e] = __ldg(tc + (size_t)p * nf + i);
            s4[e] = __ldg(ts + (size_t)p * nf + i);
          }
          cv[k] = make_float4(c4[0], c4[1], c4[2], c4[3]);
          sv[k] = make_float4(s4[0], s4[1], s4[2], s4[3]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int f = f0 + 32 * k + lane;
      if (f < total) {
        __stcs(cdst + f, cv[k]);
        __stcs(sdst + f, sv[k]);
      }
    }
  }
}

// 32 contiguous bytes (16 bf16) with one 256-bit store, evict-first.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Where the A producer thread of a tile row reads its pixels.
struct RowSrc {
  const uint8_t* base0;   // slice 0 patch origin, nullptr for rows written as zeros
  int64_t rs;             // bytes between pixel rows
  int64_t fstride;        // bytes between the frames of consecutive slices (0 for stills)
};

template <int P>
__device__ __forceinline__ RowSrc row_src(const EmbedArgs& args, const SmemHdr* hs, int r) {
  RowSrc src{nullptr, 0, 0};
  if (r < hs->tab.live) {
    const int i = find_item(hs->start, hs->tab.n, r);
    if (!tab_bit(hs->bad, i)) {
      const vitfe_item it = args.items[i];
      int tg, hh, ww;
      decode_local(r - hs->start[i], it.h, it.w, args.M, tg, hh, ww);
      const int64_t H = (int64_t)it.h * P, W = (int64_t)it.w * P;
      src.rs = W * 3;
      const bool still = (it.frames == 1);
      src.fstride = still ? 0 : H * W * 3;
      const int64_t f0 = still ? 0 : (int64_t)tg * args.T;
      src.base0 = args.pixels + it.pixel_offset + ((f0 * H + (int64_t)hh * P) * W + (int64_t)ww * P) * 3;
    }
  }
  return src;
}

// the MMA's elected lane's wait for a weight stage that had not landed at the first poll,
// out of line
__device__ __noinline__ bool wait_w_stage(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns) {
  return mbar_wait(bar, parity, abort_flag, limit_ns);
}

// the MMA's elected lane's wait for a fresh A block that was not ready at the first poll
// (cluster-scope acquire: the odd CTA's blocks are published from there), out of line
__device__ __noinline__ bool wait_a_lane(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns) {
  return mbar_wait_cl_slow(bar, parity, abort_flag, limit_ns, 0u);
}

// the first pass's warp-wide wait for a fresh A block, out of line (once per block and tile)
__device__ __noinline__ bool wait_a_block(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns) {
  return mbar_wait_warp<true>(bar, parity, abort_flag, limit_ns);
}

template <int P>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    embed_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_wf,
                 const EmbedArgs args) {
  constexpr int NBLK = nblk_of<P>();
  constexpr bool kSharedTail = w_tail_shared(3 * P * P);         // the slices' tails share an image
  constexpr int kNfb = kSharedTail ? (3 * P * P) / 64 : NBLK;    // blocks with one image per slice
  constexpr bool kLaneAWait = split_roles<P>();                  // first-pass A waits in the issuing lane
  extern __shared__ uint8_t smem_raw[];
  SmemHdr* hs = reinterpret_cast<SmemHdr*>(smem_raw);
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t tiles_base = (raw_base + (uint32_t)sizeof(SmemHdr) + 1023u) & ~1023u;
  const uint32_t a_smem = tiles_base;
  const uint32_t b_smem = tiles_base + (NBLK - ntm_blocks<P>()) * kABlockBytes;
  const int bnh = args.bn / 2;                                   // W rows per CTA per tile
  const uint32_t b_stage_bytes = (uint32_t)bnh * 128u;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const int cid = (int)cluster_id_x();
  const int ncl = (int)nclusters_x();
  volatile int* abort_flag = &hs->abort_flag;

  // ---- prologue -----------------------------------------------------------
  if (threadIdx.x == 0) {
    hs->abort_flag = 0;
    for (int j = 0; j < NBLK; ++j) {
      mbar_init(smem_u32(&hs->a_full[j]), kProducerThreads / 32 + 1);  // even CTA's warps + the odd CTA
      mbar_init(smem_u32(&hs->a_local[j]), kProducerThreads / 32);     // one arrive per producer warp
      mbar_init(smem_u32(&hs->a_empty[j]), 1);
    }
    for (int s = 0; s < args.nstage; ++s) {
      mbar_init(smem_u32(&hs->b_full[s]), 1);
      mbar_init(smem_u32(&hs->b_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&hs->acc_full[b]), 1);
      mbar_init(smem_u32(&hs->acc_empty[b]), 2 * kEpilogueThreads);
    }
    mbar_init(smem_u32(&hs->drain), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    ItemTab tab{hs->start, hs->bad, hs->still, &hs->tab};
    build_item_table(args.items, args.n_items, args.max_items, args.pixel_bytes, P, args.T, args.M,
                     args.rows, args.rope_cos != nullptr ? VITFE_ROPE_MAX_SIDE : 0x7fffffff, tab);
  }
  if (warp == mma_warp<P>()) {
    tmem_alloc_pair(smem_u32(&hs->tmem_base), (uint32_t)args.tmem_cols);
    tmem_relinquish_pair();
  }
  if (warp == w_load_warp<P>(0) && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    if (args.folded) tma_prefetch_desc(&tmap_wf);
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  // Every CTA is resident: the next call on the stream may start its prologue, A production
  // and first passes now.  This kernel reads nothing another call writes (pixels, items,
  // weights, bias, axis table); its global writes (embeddings, RoPE rows, status) wait for
  // the previous kernel of the stream to finish (grid_dep_wait in the epilogue warps and
  // before the timeout status below).
  if (threadIdx.x == 0) grid_dep_trigger();
  const uint32_t tmem = hs->tmem_base;
  // barriers of the even CTA, through the cluster shared window
  const uint32_t a_full_L = mapa_shared(smem_u32(&hs->a_full[0]), 0);
  const uint32_t b_full_L = mapa_shared(smem_u32(&hs->b_full[0]), 0);
  const uint32_t acc_empty_L = mapa_shared(smem_u32(&hs->acc_empty[0]), 0);

  // ---- roles -------------------------------------------------------------
  const int pidx = producer_index<P>(warp);
  if (pidx >= 0) {
    // A producers: this CTA's 128 rows of every pair tile, K blocks split in two halves
    const float sc[3] = {args.scale0, args.scale1, args.scale2};
    const float sh[3] = {args.shift0, args.shift1, args.shift2};
    const int row = (pidx & 3) * 32 + lane;
    const int half = pidx >> 2;
    const int rofs = (int)rank * kTileM + row;
    // this warp's lane quarter of the tensor-memory A blocks
    const uint32_t tmem_a = hs->tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    // block-ready barriers this CTA's producer warps arrive on
    const uint32_t a_ready0 = leader ? smem_u32(&hs->a_full[0]) : smem_u32(&hs->a_local[0]);
    uint32_t np = 0;
    bool ok = true;
    int u = cid;
    auto tile_of = [&](int uu) {
      int t, lo, hi;
      unit_range(args, uu, t, lo, hi);
      return t;
    };
    RowSrc cur = u < args.num_units ? row_src<P>(args, hs, tile_of(u) * kPairRows + rofs)
                                    : RowSrc{nullptr, 0, 0};
    for (; ok && u < args.num_units; u += ncl) {
      int tile, p_lo, p_hi;
      unit_range(args, u, tile, p_lo, p_hi);
      const int npu = p_hi - p_lo;   // passes of the unit
      const int kind = tile_kind(tile * kPairRows, hs, args.T);
      const int next = u + ncl;
      const RowSrc nxt = next < args.num_units ? row_src<P>(args, hs, tile_of(next) * kPairRows + rofs)
                                               : RowSrc{nullptr, 0, 0};
      if (kind != kPad) {
        // stream tiles: one production of each slice per pair of N passes
        const int nprod = (kind == kResident) ? 1 : ((npu + 1) / 2) * args.T;
        for (int q = 0; ok && q < nprod; ++q) {
          const int s = (kind == kResident) ? 0 : (q % args.T);
          const uint8_t* base = cur.base0 ? cur.base0 + cur.fstride * s : nullptr;
          if (half == 0)
            ok = produce_blocks<P, 0, NBLK / 2>(base, cur.rs, a_smem, hs, np, row, sc, sh, abort_flag,
                                                args.limit_ns, a_ready0, tmem_a);
          else
            ok = produce_blocks<P, NBLK / 2, NBLK>(base, cur.rs, a_smem, hs, np, row, sc, sh, abort_flag,
                                                   args.limit_ns, a_ready0, tmem_a);
          ++np;
        }
      }
      cur = nxt;
    }
  } else if (warp == forward_warp<P>() && !leader) {
    // every production of this CTA's A blocks, two blocks at a time in the order the MMA
    // consumes them: wait for the producer warps' local arrivals on both, then one
    // cluster-scope release arrival for the first and a relaxed one for the second (the MMA
    // acquires the first block's barrier before it waits for the second's)
    uint32_t np = 0;
    bool ok = true;
    const uint32_t a_local0 = smem_u32(&hs->a_local[0]);
    for (int u = cid; ok && u < args.num_units; u += ncl) {
      int tile, p_lo, p_hi;
      unit_range(args, u, tile, p_lo, p_hi);
      const int kind = tile_kind(tile * kPairRows, hs, args.T);
      if (kind == kPad) continue;
      const int nprod = (kind == kResident) ? 1 : ((p_hi - p_lo + 1) / 2) * args.T;
      for (int q = 0; ok && q < nprod; ++q) {
        static_assert(NBLK % 2 == 0, "blocks forwarded in pairs");
#pragma unroll 1
        for (int jj = 0; jj < NBLK; jj += 2) {
          const int j0 = blk_order<NBLK>(jj), j1 = blk_order<NBLK>(jj + 1);
          if (!mbar_wait_warp<false>(a_local0 + 8u * (uint32_t)j0, np & 1u, abort_flag, args.limit_ns) ||
              !mbar_wait_warp<false>(a_local0 + 8u * (uint32_t)j1, np & 1u, abort_flag, args.limit_ns)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_cluster(a_full_L + 8u * (uint32_t)j0);
            mbar_arrive_cluster_relaxed(a_full_L + 8u * (uint32_t)j1);
          }
          __syncwarp();
        }
        ++np;
      }
    }
  } else if (warp == w_load_warp<P>(0) || warp == w_load_warp<P>(1)) {
    // (with the failure-detection test hook set, no weight tile is ever loaded: the MMA's
    // bounded wait runs out, every role leaves on the abort flag or its own limit)
    if (lane == 0 && !args.stall_w_loads) {
      // W tiles in consumption order: one stage per step (a step = one 64-feature K block
      // of one temporal slice).  Both loading warps walk the whole sequence; this one
      // issues the stages nb with nb % kWLoaders == wl.
      const int wl = (warp == w_load_warp<P>(0)) ? 0 : 1;
      uint32_t nb = 0, stage = 0, bphase = 0;
      bool ok = true;
      for (int u = cid; ok && u < args.num_units; u += ncl) {
        int tile, p_lo, p_hi;
        unit_range(args, u, tile, p_lo, p_hi);
        const int kind = tile_kind(tile * kPairRows, hs, args.T);
        if (kind == kPad) continue;
        // folded still tiles: one slice of the folded weight per block
        const bool fold = args.folded && kind == kResident;
        const int Ts = fold ? 1 : args.T;
        const CUtensorMap* map = fold ? &tmap_wf : &tmap_w;
        // this CTA's image of (pass pg, slice sl, block j): bnh/4 rows of 512 B each; the
        // slices' one-step tails share one image (w_images)
        const int imgs = w_images(3 * P * P, Ts);
        auto img_of = [&](int pg, int sl, int j) {
          const int base = (pg * 2 + (int)rank) * imgs;
          return (kSharedTail && j == kNfb) ? base + Ts * kNfb : base + sl * kNfb + j;
        };
        auto load_image = [&](int img) {
          if ((int)(nb % (uint32_t)kWLoaders) == wl) {
            if (!mbar_wait_cl(smem_u32(&hs->b_empty[stage]), bphase ^ 1u, abort_flag, args.limit_ns)) {
              ok = false;
              return;
            }
            if (leader) mbar_arrive_expect_tx(smem_u32(&hs->b_full[stage]), 2u * b_stage_bytes);
            tma_load_2d_pair(b_smem + stage * b_stage_bytes, map, b_full_L + 8u * stage, 0, img * (bnh / 4));
          }
          ++nb;
          if (++stage == (uint32_t)args.nstage) { stage = 0; bphase ^= 1u; }
        };
        for (int p = p_lo; ok && p < p_hi;) {
          // the MMA's pairs of stream passes take, per (slice, block), both passes' images
          const int G = (kind == kStream && p + 1 < p_hi) ? 2 : 1;
          if (kind == kResident) {
            for (int jj = 0; ok && jj < NBLK; ++jj) {
              const int j = blk_order<NBLK>(jj);
              const int nsl = (kSharedTail && j == kNfb) ? 1 : Ts;   // one image holds every tail
              for (int sl = 0; ok && sl < nsl; ++sl) load_image(img_of(p, sl, j));
            }
          } else {
            for (int sl = 0; ok && sl < Ts; ++sl)
              for (int jj = 0; ok && jj < NBLK; ++jj)
                for (int g = 0; ok && g < G; ++g) load_image(img_of(p + g, sl, blk_order<NBLK>(jj)));
          }
          p += G;
        }
      }
      if (!ok) {
        if (leader) {
          // the last loads this warp issued complete on their own (its stages before nb were
          // issued; nb itself was not)
          const uint32_t nlast = nb < (uint32_t)args.nstage ? nb : (uint32_t)args.nstage;
          for (uint32_t d = 1; d <= nlast; ++d) {
            const uint32_t idx = nb - d;
            if ((int)(idx % (uint32_t)kWLoaders) != wl) continue;
            const uint32_t bar = smem_u32(&hs->b_full[idx % (uint32_t)args.nstage]);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait_cluster(bar, (idx / (uint32_t)args.nstage) & 1u) &&
                   global_timer_ns() - t0 < args.limit_ns) {
            }
          }
        } else {
          // this CTA's copies signal the even CTA's barriers: give them time to land
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 200000ull) __nanosleep(1000);
        }
      }
    }
  } else if (warp == mma_warp<P>()) {
    if (leader) {
      // The whole warp runs the issue loop, so its indices and descriptors stay warp-uniform
      // (uniform registers); one elected lane waits for each stage's weights and issues its
      // MMAs and commit, and one vote per stage reconverges the warp.  The code between issues
      // is kept minimal (descriptors at constant offsets, slow waits out of line): this one
      // warp's issue time per stage has to stay under the stage's tensor time.
      uint32_t na = 0, np = 0, stage = 0, bphase = 0;
      bool ok = true;
      const uint64_t adesc0 = sw128_desc(a_smem);
      const uint64_t bdesc0 = sw128_desc(b_smem);
      const uint64_t bstep = (uint64_t)(b_stage_bytes >> 4);
      uint64_t bd_cur = bdesc0;
      const uint32_t b_full0 = smem_u32(&hs->b_full[0]);
      const uint32_t b_empty0 = smem_u32(&hs->b_empty[0]);
      const uint32_t a_full0 = smem_u32(&hs->a_full[0]);
      const uint32_t a_empty0 = smem_u32(&hs->a_empty[0]);
      const uint32_t nstage = (uint32_t)args.nstage;
      const int T = args.T;

#define VITFE_WAIT_A(J)                                                                       \
  do {                                                                                        \
    if (!mbar_wait_warp<true>(a_full0 + 8u * (J), np & 1u, abort_flag, args.limit_ns)) ok = false; \
    if (in_tmem<P>(J)) tc_fence_after();                                                      \
  } while (0)
// One stage, issued by the elected lane alone: with AW it first waits for A block J (the
// producers' release, cluster-scope acquire); then it waits for the stage's W image (one
// poll; when the image has not landed, the bounded wait out of line), issues the K16 MMAs of
// block J (A in shared memory at descriptor ADESC, or in tensor memory) against the image
// from K16 step BOFF / 2 on, and the stage's release.  One vote ends the stage: it carries a
// timed-out wait to every lane and reconverges the warp (warp-wide polls and votes before
// the MMAs cost more issue time per stage).
#define VITFE_STEP(D, ID, J, ADESC, NK, FIRST, BOFF, AW)                                      \
  do {                                                                                        \
    const uint64_t bd_ = bd_cur + (uint64_t)(BOFF);                                           \
    bool go_ = true;                                                                          \
    if (elect_one()) {                                                                        \
      if (AW) {                                                                               \
        go_ = mbar_try_wait_cluster(a_full0 + 8u * (J), np & 1u) ||                           \
              wait_a_lane(a_full0 + 8u * (J), np & 1u, abort_flag, args.limit_ns);            \
        if (in_tmem<P>(J)) tc_fence_after();                                                  \
      }                                                                                       \
      go_ = go_ && (mbar_try_wait(b_full0 + 8u * stage, bphase) ||                            \
                    wait_w_stage(b_full0 + 8u * stage, bphase, abort_flag, args.limit_ns));   \
      if (go_) {                                                                              \
        if (in_tmem<P>(J)) {                                                                  \
          const uint32_t ta_ = tmem + tm_col<P>(J);                                           \
          umma_bf16_pair_ta((D), ta_, bd_, (ID), (FIRST) ? 0u : 1u);                          \
          if ((NK) > 1) umma_bf16_pair_ta((D), ta_ + 8u, bd_ + 2u, (ID), 1u);                \
          if ((NK) > 2) umma_bf16_pair_ta((D), ta_ + 16u, bd_ + 4u, (ID), 1u);               \
          if ((NK) > 3) umma_bf16_pair_ta((D), ta_ + 24u, bd_ + 6u, (ID), 1u);               \
        } else {                                                                              \
          umma_bf16_pair((D), (ADESC), bd_, (ID), (FIRST) ? 0u : 1u);                         \
          if ((NK) > 1) umma_bf16_pair((D), (ADESC) + 2u, bd_ + 2u, (ID), 1u);               \
          if ((NK) > 2) umma_bf16_pair((D), (ADESC) + 4u, bd_ + 4u, (ID), 1u);               \
          if ((NK) > 3) umma_bf16_pair((D), (ADESC) + 6u, bd_ + 6u, (ID), 1u);               \
        }                                                                                     \
        umma_commit_pair(b_empty0 + 8u * stage);                                              \
      }                                                                                       \
    }                                                                                         \
    if (!__all_sync(0xffffffffu, go_)) ok = false;                                            \
    if (++stage == nstage) {                                                                  \
      stage = 0;                                                                              \
      bphase ^= 1u;                                                                           \
      bd_cur = bdesc0;                                                                        \
    } else {                                                                                  \
      bd_cur += bstep;                                                                        \
    }                                                                                         \
  } while (0)

// one stage holding the NS temporal slices' one-step tails of block kNfb: each slice's K16
// MMA against the same A block, slice s at K16 step s of the image (never a pass's first
// MMA); AW as for VITFE_STEP
#define VITFE_STEP_TAILS(D, ID, ADESC, NS, AW)                                                \
  do {                                                                                        \
    const uint64_t bd_ = bd_cur;                                                              \
    bool go_ = true;                                                                          \
    if (elect_one()) {                                                                        \
      if (AW) {                                                                               \
        go_ = mbar_try_wait_cluster(a_full0 + 8u * kNfb, np & 1u) ||                          \
              wait_a_lane(a_full0 + 8u * kNfb, np & 1u, abort_flag, args.limit_ns);           \
        if (in_tmem<P>(kNfb)) tc_fence_after();                                               \
      }                                                                                       \
      go_ = go_ && (mbar_try_wait(b_full0 + 8u * stage, bphase) ||                            \
                    wait_w_stage(b_full0 + 8u * stage, bphase, abort_flag, args.limit_ns));   \
      if (go_) {                                                                              \
        for (int s_ = 0; s_ < (NS); ++s_) umma_bf16_pair((D), (ADESC), bd_ + 2u * (uint64_t)s_, (ID), 1u); \
        umma_commit_pair(b_empty0 + 8u * stage);                                              \
      }                                                                                       \
    }                                                                                         \
    if (!__all_sync(0xffffffffu, go_)) ok = false;                                            \
    if (++stage == nstage) {                                                                  \
      stage = 0;                                                                              \
      bphase ^= 1u;                                                                           \
      bd_cur = bdesc0;                                                                        \
    } else {                                                                                  \
      bd_cur += bstep;                                                                        \
    }                                                                                         \
  } while (0)

      for (int u = cid; ok && u < args.num_units; u += ncl) {
        int tile, p_lo, p_hi;
        unit_range(args, u, tile, p_lo, p_hi);
        const int kind = tile_kind(tile * kPairRows, hs, args.T);
        if (kind == kPad) continue;
        for (int p = p_lo; ok && p < p_hi;) {
          // a stream tile's N passes go in pairs, one accumulator each, so that every
          // production of its A (both temporal slices) feeds two passes
          const int G = (kind == kStream && p + 1 < p_hi) ? 2 : 1;
          for (int g = 0; ok && g < G; ++g) {
            const uint32_t n_ = na + (uint32_t)g;
            if (!mbar_wait_warp<true>(smem_u32(&hs->acc_empty[n_ & 1u]), ((n_ >> 1) & 1u) ^ 1u, abort_flag,
                                      args.limit_ns))
              ok = false;
          }
          if (!ok) break;
          tc_fence_after();
          const uint32_t buf = na & 1u;
          const uint32_t idesc = idesc_bf16(kPairRows, min(args.bn, args.N - p * args.bn));
          const uint32_t d_tmem = tmem + buf * (uint32_t)args.bn;
          if (kind == kResident) {
            // one resident slice of A feeds every temporal slice of W (one folded slice)
            const int Ts = args.folded ? 1 : T;
#pragma unroll
            for (int jj = 0; jj < NBLK; ++jj) {
              const int j = blk_order<NBLK>(jj);
              // the unit's first pass meets the fresh A: each block is waited for before its
              // first stage, by the issuing lane (patch 14) or by the whole warp (patch 16, where
              // the lane's wait measured slower)
              if (!kLaneAWait && p == p_lo) {
                if (!wait_a_block(a_full0 + 8u * (uint32_t)j, np & 1u, abort_flag, args.limit_ns)) ok = false;
                if (in_tmem<P>(j)) tc_fence_after();
              }
              if (!ok) break;
              const bool aw = kLaneAWait && p == p_lo;
              const uint64_t ad = adesc0 + (uint64_t)(smem_slot<P>(j) * (kABlockBytes >> 4));
              if (kSharedTail && j == kNfb) {
                VITFE_STEP_TAILS(d_tmem, idesc, ad, Ts, aw);
              } else {
                for (int sl = 0; ok && sl < Ts; ++sl)
                  VITFE_STEP(d_tmem, idesc, j, ad, ksteps_of<P>(j), j == 0 && sl == 0, 0u, aw && sl == 0);
              }
              if (!ok) break;
              if (p == p_hi - 1) {
                if (elect_one()) umma_commit_pair(a_empty0 + 8u * j);
                __syncwarp();
              }
            }
          } else {
            // the pair's second pass (G == 2): the other accumulator
            const uint32_t idesc1 = idesc_bf16(kPairRows, min(args.bn, args.N - (p + 1) * args.bn));
            const uint32_t d_tmem1 = tmem + (buf ^ 1u) * (uint32_t)args.bn;
            for (int sl = 0; ok && sl < T; ++sl) {
#pragma unroll
              for (int jj = 0; jj < NBLK; ++jj) {
                const int j = blk_order<NBLK>(jj);
                const uint64_t ad = adesc0 + (uint64_t)(smem_slot<P>(j) * (kABlockBytes >> 4));
                VITFE_WAIT_A(j);
                // one copy of the issue code for both passes (code size: the issue loop is
                // sensitive to instruction fetch)
#pragma unroll 1
                for (int g = 0; ok && g < G; ++g) {
                  VITFE_STEP(g ? d_tmem1 : d_tmem, g ? idesc1 : idesc, j, ad, ksteps_of<P>(j), sl == 0 && j == 0,
                             (kSharedTail && j == kNfb) ? 2u * (uint32_t)sl : 0u, false);
                }
                if (!ok) break;
                if (elect_one()) umma_commit_pair(a_empty0 + 8u * j);
                __syncwarp();
              }
              ++np;   // one slice production consumed
            }
          }
          if (!ok) break;
          if (elect_one()) {
            for (int g = 0; g < G; ++g) umma_commit_pair(smem_u32(&hs->acc_full[(na + (uint32_t)g) & 1u]));
          }
          __syncwarp();
          na += (uint32_t)G;
          p += G;
        }
        if (kind == kResident) ++np;
      }
#undef VITFE_STEP_TAILS
#undef VITFE_STEP
#undef VITFE_WAIT_A
      if (!ok) {
        // the elected lane issued every MMA: its commit covers them all
        if (elect_one()) umma_commit_pair(smem_u32(&hs->drain));
        __syncwarp();
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait_cluster(smem_u32(&hs->drain), 0u) && global_timer_ns() - t0 < args.limit_ns) {
        }
      }
    }
  } else if (epilogue_warp<P>(warp)) {
    // epilogue: lane quarter q = warp % 4 of this CTA's accumulator rows
    const int q = warp & 3;
    const int rloc = (int)rank * kTileM + q * 32 + lane;
    const bool out32 = (reinterpret_cast<uintptr_t>(args.out) & 31u) == 0;
    uint32_t na = 0;
    bool ok = true;
    // the first global write of this call: after the previous kernel of the stream
    grid_dep_wait();
    if (blockIdx.x == 0 && q == 0 && lane == 0 && args.status != nullptr) {
      args.status[0] = hs->tab.code;
      args.status[1] = hs->tab.bad_item;
    }
    for (int u = cid; ok && u < args.num_units; u += ncl) {
      int tile, p_lo, p_hi;
      unit_range(args, u, tile, p_lo, p_hi);
      const int r0 = tile * kPairRows;
      const int kind = tile_kind(r0, hs, args.T);
      const int r = r0 + rloc;
      const bool in_bucket = r < args.rows;
      bool valid = false;
      int hp = -1, wp = -1;
      if (r < hs->tab.live) {
        const int i = find_item(hs->start, hs->tab.n, r);
        valid = !tab_bit(hs->bad, i);
        if (valid && args.rope_cos != nullptr) {
          const vitfe_item it = args.items[i];
          int tg;
          decode_local(r - hs->start[i], it.h, it.w, args.M, tg, hp, wp);
        }
      }
      const int rope_wbase = r0 + (int)rank * kTileM + q * 32;
      __nv_bfloat16* orow = args.out + (size_t)r * (size_t)args.N;
      // this unit's columns; the unit holding pass 0 also writes the rows' RoPE
      const bool rope_unit = args.rope_cos != nullptr && p_lo == 0;
      if (kind == kPad) {
        if (in_bucket) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          const int c_hi = min(args.N, p_hi * args.bn);
          for (int c = p_lo * args.bn; c < c_hi; c += 8) *reinterpret_cast<uint4*>(orow + c) = z;
        }
        if (rope_unit) rope_rows(args, rope_wbase, hp, wp, lane);
        continue;
      }
      // the RoPE rows of this warp's 32 tile rows go out after the second pass's accumulator:
      // the producers are idle then (they fill the next tile's A during the first and last
      // passes) and the epilogue waits for the next accumulator anyway
      const int rope_pass = p_hi - p_lo > 1 ? p_lo + 1 : p_lo;
      for (int p = p_lo; p < p_hi; ++p) {
        const uint32_t buf = na & 1u;
        // warp-uniform wait: tcgen05.ld below (and the RoPE rows' shuffles) need the whole warp
        if (!mbar_wait_warp<true>(smem_u32(&hs->acc_full[buf]), (na >> 1) & 1u, abort_flag, args.limit_ns, 64)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int npw = min(args.bn, args.N - p * args.bn);
        // fewer L1 wavefronts for the stores (the lanes swap halves, below) where the drain
        // overlaps the next pass of a resident tile; where the drain is on the critical path
        // (a unit's last pass, stream tiles' pass pairs) the shuffles would lengthen it
        const bool swap = out32 && kind == kResident && p + 1 < p_hi;
        for (int c0 = 0; c0 < npw; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + buf * (uint32_t)args.bn + (uint32_t)c0, v);
          tmem_wait_ld();
          const int n0 = p * args.bn + c0;
          uint32_t pk[16];
          const float4* bias4 = reinterpret_cast<const float4*>(args.bias + n0);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 bv = __ldg(bias4 + e4);
            __nv_bfloat162 b0 = __floats2bfloat162_rn(__uint_as_float(v[4 * e4]) + bv.x,
                                                      __uint_as_float(v[4 * e4 + 1]) + bv.y);
            __nv_bfloat162 b1 = __floats2bfloat162_rn(__uint_as_float(v[4 * e4 + 2]) + bv.z,
                                                      __uint_as_float(v[4 * e4 + 3]) + bv.w);
            pk[2 * e4] = valid ? *reinterpret_cast<uint32_t*>(&b0) : 0u;
            pk[2 * e4 + 1] = valid ? *reinterpret_cast<uint32_t*>(&b1) : 0u;
          }
          if (swap) {
            // Lanes 2m and 2m+1 swap halves, so that each 256-bit store covers 64 contiguous
            // bytes of a row (16 rows an instruction) rather than 32 bytes of 32 rows: the first
            // store writes the even row of the pair, the second the odd one, the even lane the
            // first 32 bytes of each and the odd lane the last 32.
            const uint32_t odd = (uint32_t)lane & 1u;
            uint32_t d1[8], d2[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? pk[w] : pk[8 + w], 1);
              d1[w] = odd ? recv : pk[w];
              d2[w] = odd ? pk[8 + w] : recv;
            }
            const int re = r - (int)odd;                 // the pair's even row
            __nv_bfloat16* dst = args.out + (size_t)re * (size_t)args.N + n0 + 16 * (int)odd;
            if (re < args.rows) st_global_v8(dst, d1);
            if (re + 1 < args.rows) st_global_v8(dst + args.N, d2);
          } else if (in_bucket) {
            __nv_bfloat16* dst = orow + n0;
            if (out32) {
              st_global_v8(dst, pk);
              st_global_v8(dst + 16, pk + 8);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int e = 0; e < 4; ++e) __stcs(d4 + e, make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]));
            }
          }
        }
        tc_fence_before();
        mbar_arrive_cluster(acc_empty_L + 8u * buf);
        ++na;
        if (rope_unit && p == rope_pass) rope_rows(args, rope_wbase, hp, wp, lane);
      }
    }
  }

  // ---- teardown ------------------------------------------------------------
  __syncwarp();
  // a producer that left on a timeout may still have tensor-memory stores in flight
  if (ntm_blocks<P>() > 0 && pidx >= 0) tmem_wait_st();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == mma_warp<P>()) tmem_dealloc_pair(tmem, (uint32_t)args.tmem_cols);
  if (threadIdx.x == 0 && hs->abort_flag && args.status != nullptr) {
    grid_dep_wait();
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
  // implemented: patch 14 or 16 (Qwen2/2.5-VL and Qwen3-VL); hidden a multiple of 64
  // (each epilogue warp stores whole 32-column groups of its half of a pass)
  if (!(c.P == 14 || c.P == 16) || (c.N % 64) != 0) return cudaSuccess;
  int max_optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c.device);
  if (e != cudaSuccess) return e;
  // widest N tile first (fewest MMA issues per flop; patch 16: at most 192, so that two
  // accumulators leave tensor-memory room for its A blocks); a stage holds this CTA's half
  // of one W tile, and at least two stages must fit beside the shared-memory A blocks
  const int ntm = c.P == 16 ? ntm_blocks<16>() : ntm_blocks<14>();
  for (int bn : {c.P == 16 ? 192 : 256, 128}) {
    if (bn > c.N && bn != 128) continue;
    const int b = bn < c.N ? bn : c.N;
    for (int nst = 8; nst >= 2 && !c.embed_ok; --nst) {
      const size_t need = embed_smem_bytes(c.nblk - ntm, b / 2, nst);
      if (need <= (size_t)max_optin) {
        c.bn = b;
        c.nstage = nst;
        c.embed_smem = need;
        c.embed_ok = true;
      }
    }
    if (c.embed_ok) break;
  }
  if (!c.embed_ok) return cudaSuccess;
  const void* fn = (c.P == 14) ? (const void*)embed_kernel<14> : (const void*)embed_kernel<16>;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.embed_smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (c.sm_count / 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = c.embed_smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int ncl = 0;
  e = cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg);
  if (e != cudaSuccess) return e;
  c.max_clusters = ncl > 0 ? ncl : 1;
  return cudaSuccess;
}

cudaError_t launch_embed(const Ctx& c, const uint8_t* pixels, int64_t pixel_bytes,
                         const vitfe_item* items, const int32_t* n_items, int max_items,
                         int64_t rows, void* out, int32_t* status, cudaStream_t s, const float* rope_tab,
                         int rope_nf, float* rope_cos, float* rope_sin, bool folded) {
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
  a.bn = c.bn;
  a.nstage = c.nstage;
  a.npass = (c.N + c.bn - 1) / c.bn;
  a.tmem_cols = 32;
  while (a.tmem_cols < 2 * c.bn) a.tmem_cols <<= 1;
  if (c.P == 16) a.tmem_cols = 512;   // A blocks from column kTmemACol
  a.num_tiles = (int)((rows + kPairRows - 1) / kPairRows);
  // The tiles of a last round that would leave CTA pairs idle (all tiles of a batch with
  // fewer tiles than pairs) have their N passes spread over several pairs, each of which
  // produces the tile's A itself: a round of few tiles is then not one pair's five passes
  // in a row.  The passes of a tile give the same results on whichever pair runs them.
  {
    const int R = c.max_clusters;
    const int rem = a.num_tiles % R;
    int split = rem > 0 ? R / rem : 1;
    if (split > a.npass) split = a.npass;
    if (split < 1) split = 1;
    a.ppu = (a.npass + split - 1) / split;
    a.split = (a.npass + a.ppu - 1) / a.ppu;
    a.whole_tiles = a.num_tiles - rem;
    a.num_units = a.whole_tiles + rem * a.split;
  }
  a.limit_ns = c.wait_limit_ns;
  a.stall_w_loads = c.test_stall_w_loads ? 1 : 0;
  a.rope_tab = rope_tab;
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.rope_nf = rope_nf;
  a.folded = folded ? 1 : 0;
  int pairs = a.num_units < c.max_clusters ? a.num_units : c.max_clusters;
  if (pairs < 1) pairs = 1;
  const int grid = 2 * pairs;
  // programmatic stream serialization: the launch may begin while the previous kernel of the
  // stream finishes (the kernel orders its own writes after it)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = c.embed_smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (c.P == 14) return cudaLaunchKernelEx(&cfg, embed_kernel<14>, c.tmap_w, c.tmap_wf, a);
  return cudaLaunchKernelEx(&cfg, embed_kernel<16>, c.tmap_w, c.tmap_wf, a);
}

}  // namespace vitfe
