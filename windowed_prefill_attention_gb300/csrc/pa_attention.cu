// Attention kernel of the windowed prefill attention over a paged int8 KV pool
// (sm_103a): a persistent, warp-specialised tcgen05 pipeline.
//
// The method ("int8 tensor-core prefill attention", sections "Summary" and
// "Why the attention, and why tensor cores"): the query quantised per row in
// a fused prologue; QK^T on the tensor cores over K codes read from the paged
// pool; the per-row Q, per-token K and softmax scales applied to the integer-
// valued scores; the online-softmax recurrence; the per-token V scale folded
// into P before P is quantised per row; PV on the tensor cores; masked blocks
// never visited.  The int8 codes travel in fp16 containers (tcgen05.mma
// kind::f16), which hold them exactly.
//
// One CTA per SM walks the longest-first unit list with stride gridDim.x.  A
// unit is 128 query rows of one kv head (pa_tiles.cuh).  Roles:
//   warp 0        TMA producer: K tiles into a 3-slot ring, V^T tiles and the
//                 tile's K/V scales into another 3-slot ring
//   warp 1        TMEM allocator and the single MMA-issuing thread:
//                 QK^T(j+1) is issued before PV(j), so the tensor core works on
//                 the next scores while the softmax handles the current ones
//   warps 4-11    softmax: one query row per thread (TMEM lane = row), two
//                 warps per lane quadrant, each owning half of the key columns
//   warps 12-15   Q prologue of the next unit and epilogue of the previous one
// TMEM (512 columns): O fp32 [0,256), Q fp16 pairs [256,384), S0/S1 fp32
// [384,448)/[448,512); P (fp16 pairs) overwrites the first half of its S.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kThreads = 512;
constexpr int kSlots = 3;                              // depth of the K ring and of the V ring
constexpr int kKTileBytes = kTileKeys * kHeadDim * 2;  // 32 KB: 4 regions of 64 keys x 128 B
constexpr int kVTileBytes = kHeadDim * kTileKeys * 2;  // 32 KB: 256 dims x 128 B
// Shared memory, offsets from a 1024-byte aligned base.
constexpr int kSmK = 0;
constexpr int kSmV = kSmK + kSlots * kKTileBytes;
constexpr int kSmScale = kSmV + kSlots * kVTileBytes;  // per slot: ks[64] (K ring) then vs[64] (V ring)
constexpr int kSmRows = kSmScale + kSlots * 512;       // c[2][128], l[2][2][128], sp[2][128] floats
constexpr int kSmXchg = kSmRows + 8 * kRows * 4;       // softmax pair exchange: 2 x [2][2][128] floats
constexpr int kSmBars = kSmXchg + 8 * kRows * 4;
enum : int {
  B_KFULL = 0, B_KEMPTY = 3, B_VFULL = 6, B_VEMPTY = 9, B_SFULL = 12, B_PFULL = 14,
  B_QFULL = 16, B_QEMPTY = 17, B_OFULL = 18, B_OEMPTY = 19, B_STATS = 20 /* two, by unit parity */,
  B_STALL = 22, B_DRAIN = 23, kNumBars = 24
};
constexpr float kLift = 6.f;   // a unit's first reference sits 2^kLift above its first tile's max
constexpr float kLazy = 14.f;  // the softmax reference moves when a row max grows by more than 2^kLazy;
                               // P' = p * v_scale * 2^-ev then stays below 2^14, inside the fp16 range
constexpr int kSmTmemSlot = kSmBars + kNumBars * 8;
constexpr int kAttnSmem = kSmTmemSlot + 16 + 1024;  // + alignment slack
static_assert(kAttnSmem <= 227 * 1024, "shared memory budget");

constexpr uint32_t kTmO = 0;
constexpr uint32_t kTmQ = 256;
constexpr uint32_t kTmS = 384;
constexpr uint64_t kDrainNs = 200000000ull;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
// e with 2^(e-1) <= x < 2^e, clamped to [-100, 100]; 0 for x <= 0.
__device__ __forceinline__ int pow2_ceil_exp(float x) {
  if (!(x > 0.f)) return 0;
  const int eb = (int)((__float_as_uint(x) >> 23) & 0xff);
  return imax(-100, imin(100, eb - 126));
}

struct Ctx {
  uint32_t sbase;  // shared address of the aligned base
  uint32_t tb;     // TMEM base address
  WaitCtl wc;
  __device__ uint32_t bar(int i) const { return sbase + kSmBars + 8 * i; }
  // Bounded wait by all 32 lanes of a warp with one outcome for the warp, so
  // that the warp-collective tcgen05.ld/st and __syncwarp that follow never
  // see a diverged warp, also when a wait runs out.
  __device__ bool warp_wait(int i, uint32_t parity, int site) const {
    const bool r = mbar_wait(bar(i), parity, wc, site);
    return __all_sync(0xffffffffu, r);
  }
};

// ------------------------------------------------------------------ producer
__device__ __forceinline__ void role_producer(const AttnParams& p, const AttnMaps& m, const Ctx& c) {
  uint32_t kc = 0, vc = 0;  // loads issued into the K ring and the V ring
  bool ok = true;
  for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const UnitGeom ug = unit_geom(un.t0, p.TQ, sg, p.S, p.W);
    for (int j = 0; j < ug.n_tiles; ++j) {
      const TileGeom tg = tile_geom(ug, j, p.S, p.W);
      const int crow = logical_block_row(sg, tg.kb0);
      {
        const int s = kc % kSlots;
        const uint32_t ph = (kc / kSlots) & 1;
        if (!(ok = mbar_wait(c.bar(B_KEMPTY + s), ph ^ 1, c.wc, 10))) break;
        const uint32_t fb = c.bar(B_KFULL + s);
        const uint32_t sbytes = (uint32_t)(tg.nb * kPage * 4);
        mbar_expect_tx(fb, kKTileBytes + sbytes);
        const uint32_t dst = c.sbase + kSmK + s * kKTileBytes;
        for (int r = 0; r < 4; ++r) tma_load_3d(dst + r * 8192, &m.k, fb, r * 64, crow, un.g);
        bulk_load(c.sbase + kSmScale + s * 512, p.ks + (size_t)un.g * p.n_tok_cap + crow, sbytes, fb);
        ++kc;
      }
      {
        const int s = vc % kSlots;
        const uint32_t ph = (vc / kSlots) & 1;
        if (!(ok = mbar_wait(c.bar(B_VEMPTY + s), ph ^ 1, c.wc, 11))) break;
        const uint32_t fb = c.bar(B_VFULL + s);
        const uint32_t sbytes = (uint32_t)(tg.nb * kPage * 4);
        mbar_expect_tx(fb, kVTileBytes + sbytes);
        tma_load_3d(c.sbase + kSmV + s * kVTileBytes, &m.v, fb, crow, 0, un.g);
        bulk_load(c.sbase + kSmScale + s * 512 + 256, p.vs + (size_t)un.g * p.n_tok_cap + crow, sbytes, fb);
        ++vc;
      }
    }
  }
  // every issued copy lands before the CTA may exit: the last load into each
  // slot was load number kc-1-i (K) / vc-1-i (V) for i < kSlots
  for (uint32_t i = 0; i < (uint32_t)kSlots; ++i) {
    if (kc > i) (void)mbar_wait_drain(c.bar(B_KFULL + (kc - 1 - i) % kSlots), ((kc - 1 - i) / kSlots) & 1, kDrainNs);
    if (vc > i) (void)mbar_wait_drain(c.bar(B_VFULL + (vc - 1 - i) % kSlots), ((vc - 1 - i) / kSlots) & 1, kDrainNs);
  }
}

// ------------------------------------------------------------------ MMA issuer
__device__ __forceinline__ void role_mma(const AttnParams& p, const Ctx& c) {
  uint32_t tc = 0;  // global tile counter: K slot, V slot and S buffer of every tile
  int k_unit = 0;
  bool ok = true;
  const uint32_t id_pv = idesc_f16(kRows, kHeadDim, false, false);
  for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++k_unit) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const UnitGeom ug = unit_geom(un.t0, p.TQ, sg, p.S, p.W);
    const int n = ug.n_tiles;
    if (!(ok = mbar_wait(p.debug_stall ? c.bar(B_STALL) : c.bar(B_QFULL), k_unit & 1, c.wc, 20))) break;
    tc_fence_after();
    for (int j = 0; j <= n && ok; ++j) {
      if (j < n) {  // S(j) = Q K(j)^T
        const uint32_t t = tc + j;
        const TileGeom tg = tile_geom(ug, j, p.S, p.W);
        if (!(ok = mbar_wait(c.bar(B_KFULL + t % kSlots), (t / kSlots) & 1, c.wc, 21))) break;
        tc_fence_after();
        const uint32_t kaddr = c.sbase + kSmK + (t % kSlots) * kKTileBytes;
        const uint32_t d = c.tb + kTmS + (t & 1) * kTileKeys;
        const uint32_t id = idesc_f16(kRows, tg.nb * kPage, false, false);
        // k-step s reads K bytes at kaddr + (s/4)*8192 + (s%4)*32: only the
        // descriptor's start-address field (address >> 4) moves
        const uint64_t kd0 = sdesc_k_sw128(kaddr);
#pragma unroll
        for (int s = 0; s < kHeadDim / 16; ++s)
          mma_ts(d, c.tb + kTmQ + 8 * s, kd0 + (uint64_t)(((s >> 2) * 8192 + (s & 3) * 32) >> 4), id, s > 0);
        mma_commit(c.bar(B_SFULL + (t & 1)));  // also frees K slot t: the softmax passes it on
        if (j == n - 1) mma_commit(c.bar(B_QEMPTY));
      }
      if (j >= 1) {  // O (+)= P(j-1) V(j-1)
        const int jj = j - 1;
        const uint32_t t = tc + jj;
        const TileGeom tg = tile_geom(ug, jj, p.S, p.W);
        if (!(ok = mbar_wait(c.bar(B_PFULL + (t & 1)), (t >> 1) & 1, c.wc, 22))) break;
        if (!(ok = mbar_wait(c.bar(B_VFULL + t % kSlots), (t / kSlots) & 1, c.wc, 23))) break;
        if (jj == 0 && k_unit > 0 && !(ok = mbar_wait(c.bar(B_OEMPTY), (k_unit - 1) & 1, c.wc, 24))) break;
        tc_fence_after();
        const uint32_t vaddr = c.sbase + kSmV + (t % kSlots) * kVTileBytes;
        const uint32_t a = c.tb + kTmS + (t & 1) * kTileKeys;
        const uint64_t vd0 = sdesc_k_sw128(vaddr);
        for (int s = 0; s < tg.nb; ++s)
          mma_ts(c.tb + kTmO, a + 8 * s, vd0 + (uint64_t)(2 * s), id_pv, (jj > 0 || s > 0) ? 1u : 0u);
        mma_commit(c.bar(B_VEMPTY + t % kSlots));  // V slot t free; O holds PV up to tile t
        if (jj == n - 1) mma_commit(c.bar(B_OFULL));
      }
    }
    tc += n;
  }
  // every issued MMA completes before TMEM is freed
  mma_commit(c.bar(B_DRAIN));
  (void)mbar_wait_drain(c.bar(B_DRAIN), 0, kDrainNs);
}

// ------------------------------------------------------------------ softmax
// Two warps per TMEM lane quadrant: warp half h owns key columns [32h, 32h+32)
// of every 64-key tile for the same 32 rows.  The pair agrees on each row's
// running maximum through shared memory, so both halves use one reference and
// their P', partial sums and halves of the O rescale add up exactly.
__device__ __forceinline__ void role_softmax(const AttnParams& p, const Ctx& c, uint8_t* sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3;              // lane quadrant
  const int h = (warp - 4) >> 2;        // column half
  const int r = qd * 32 + lane;         // query row = TMEM lane
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  float* c_rows = reinterpret_cast<float*>(sm + kSmRows);
  float* l_rows = c_rows + 2 * kRows;           // [unit parity][half][row]
  float* sp_rows = c_rows + 6 * kRows;          // [unit parity][row]
  float* xbuf = reinterpret_cast<float*>(sm + kSmXchg);  // [tile parity][half][row] row maxima
  float* pbuf = xbuf + 4 * kRows;                        // [tile parity][half][row] P' maxima (u8 grid)
  const bool u8 = p.p_mode == 1;
  uint32_t tc = 0;
  int k_unit = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++k_unit) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const UnitGeom ug = unit_geom(un.t0, p.TQ, sg, p.S, p.W);
    const int n = ug.n_tiles;
    const int t_row = un.t0 + r / p.G;
    const float ev = (float)pow2_ceil_exp(__uint_as_float(p.vsmax[un.seq * p.HKV + un.g]));
    // both warps of the pair agree before entering the unit's tiles
    ok = bar_red_and(1 + qd, 64, c.warp_wait(B_QFULL, k_unit & 1, 30));
    if (!ok) break;
    // s_q * sm_scale * log2(e), kept positive so that -inf scores stay -inf
    const float c_row = fmaxf(c_rows[(k_unit & 1) * kRows + r], 1e-30f);
    float m_run = -INFINITY, l_run = 0.f, sp_prev = 1.f;
    for (int j = 0; j < n; ++j) {
      const uint32_t t = tc + j;
      const TileGeom tg = tile_geom(ug, j, p.S, p.W);
      // Every path through a tile passes the pair barrier the same number of
      // times, so a wait that runs out in one warp cannot strand its partner.
      bool okl = c.warp_wait(B_SFULL + (t & 1), (t >> 1) & 1, 31);
      // the K scales landed with K slot t, which QK(t) already consumed; wait on
      // that slot's barrier too so this warp observes the copy itself (the
      // phase cannot move on before this warp releases the slot below)
      okl = okl && c.warp_wait(B_KFULL + t % kSlots, (t / kSlots) & 1, 34);
      const uint32_t sd = c.tb + lane_off + kTmS + (t & 1) * kTileKeys;
      const uint32_t sc = c.sbase + kSmScale + (t % kSlots) * 512 + 128 * h;  // this half's ks; vs at +256
      float y[32];
      float my = -INFINITY;
      if (okl) {
        tc_fence_after();
        uint32_t sa[32];
        tmem_ld32(sd + 32 * h, sa);
        tmem_wait_ld(sa);
        // y = S * k_scale (masked: -inf), and this half's row maximum
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (!tg.needs_mask && tg.nb == kTileBlocks) {  // full tile, every row sees every key
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 k4 = lds_f32x4(sc + 16 * q4);
            const float kq[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = 4 * q4 + e;
              y[q] = __uint_as_float(sa[q]) * kq[e];
              m4[e] = fmaxf(m4[e], y[q]);
            }
          }
        } else {
          const uint32_t vis = (uint32_t)(visible_columns(tg, t_row, p.S, p.W) >> (32 * h));
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 k4 = lds_f32x4(sc + 16 * q4);
            const float kq[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = 4 * q4 + e;
              y[q] = ((vis >> q) & 1u) ? __uint_as_float(sa[q]) * kq[e] : -INFINITY;
              m4[e] = fmaxf(m4[e], y[q]);
            }
          }
        }
        my = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c_row;  // log2 units
      }
      // this warp is done with K slot t (QK(t) finished before S(t) was complete)
      __syncwarp();
      if (okl && lane == 0) mbar_arrive(c.bar(B_KEMPTY + t % kSlots));
      // the reference moves only when some row's max grew by more than 2^kLazy
      const bool grow = okl && (m_run == -INFINITY || my > m_run + kLazy);
      float alpha = 1.f;
      if (bar_red_popc(1 + qd, 64, grow || !okl) != 0) {
        float* xb = xbuf + (t & 1) * 2 * kRows;
        xb[h * kRows + r] = my;
        if (!bar_red_and(1 + qd, 64, okl)) {
          ok = false;
          break;
        }
        const float mx = fmaxf(xb[r], xb[kRows + r]);
        if (m_run == -INFINITY) {
          m_run = mx == -INFINITY ? mx : mx + kLift;  // alpha irrelevant: nothing accumulated yet
          alpha = 0.f;
        } else if (mx > m_run + kLazy) {
          alpha = ex2_approx(m_run - mx);
          m_run = mx;
        }
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run + ev;
      // the V scales of tile t arrive with the V tile; a wait that runs out
      // leaves the loop after the next group barrier, like the others
      if (!c.warp_wait(B_VFULL + t % kSlots, (t / kSlots) & 1, 32)) okl = false;
      // p = 2^(y c - mref); P' = p * v_scale (V scale folded into P)
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 v4 = lds_f32x4(sc + 256 + 16 * q4);
        const float vq[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = 4 * q4 + e;
          const float pj = ex2_approx(fmaf(y[q], c_row, -mref));
          s4[e] += pj;
          y[q] = pj * vq[e];
        }
      }
      l_run = l_run * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
      float corr = alpha;
      if (u8) {  // P' per row on the u8 grid over the whole tile, scale max/255
        float pm = 0.f;
#pragma unroll
        for (int q = 0; q < 32; ++q) pm = fmaxf(pm, y[q]);
        float* pb = pbuf + (t & 1) * 2 * kRows;
        pb[h * kRows + r] = pm;
        bar_red_and(1 + qd, 64, true);
        const float pmax = fmaxf(pb[r], pb[kRows + r]);
        const float sp = pmax > 0.f ? __fdiv_rn(pmax, 255.f) : sp_prev;
        const float inv = pmax > 0.f ? __fdiv_rn(255.f, pmax) : 0.f;
#pragma unroll
        for (int q = 0; q < 32; ++q) y[q] = rintf(y[q] * inv);
        corr = alpha * __fdiv_rn(sp_prev, sp);
        sp_prev = sp;
      }
      uint32_t pk[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) pk[q] = pack_half2(y[2 * q], y[2 * q + 1]);
      tmem_st16(sd + 16 * h, pk);
      // O holds PV up to tile j-1 once that MMA is done; rescale this half in
      // place.  A wait that runs out skips the rescale without leaving the
      // loop: the error word then fails the next tile's pair barrier for both.
      if (j > 0 && __any_sync(0xffffffffu, corr != 1.f) &&
          c.warp_wait(B_VEMPTY + (t - 1) % kSlots, ((t - 1) / kSlots) & 1, 33)) {
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          const uint32_t oa = c.tb + lane_off + kTmO + 128 * h + cc * 32;
          tmem_ld32(oa, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * corr);
          tmem_st32(oa, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(B_PFULL + (t & 1)));
    }
    if (!ok) break;
    tc += n;
    l_rows[(k_unit & 1) * 2 * kRows + h * kRows + r] = l_run;
    if (h == 0) sp_rows[(k_unit & 1) * kRows + r] = sp_prev;
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(B_STATS + (k_unit & 1)));
  }
  tmem_wait_st();
}

// ------------------------------------------------------------------ prologue / epilogue
struct RowInfo {
  int t_row, h_row;
  bool valid;
  size_t off;  // element offset of the row in q / out
};

__device__ __forceinline__ RowInfo row_info(const AttnParams& p, const Unit& un, const SeqGeom& sg, int r) {
  RowInfo ri;
  ri.t_row = un.t0 + r / p.G;
  ri.h_row = un.g * p.G + r % p.G;
  ri.valid = ri.t_row >= sg.q_start && ri.t_row < sg.q_start + sg.n_q;
  ri.off = ri.valid ? ((size_t)(sg.q_off + ri.t_row - sg.q_start) * p.HQ + ri.h_row) * kHeadDim : 0;
  return ri;
}

// First pass of the Q prologue: the row's absolute maximum.  It touches no
// TMEM, so it runs before the previous unit's Q is released and leaves the
// row in L1/L2 for the second pass.
__device__ __forceinline__ float q_absmax(const AttnParams& p, const RowInfo& ri) {
  const uint4* src = reinterpret_cast<const uint4*>(p.q + ri.off);
  float absmax = 0.f;
  if (ri.valid) {
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const uint4 v = __ldg(src + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        absmax = fmaxf(absmax, fabsf(__uint_as_float(w[e] << 16)));
        absmax = fmaxf(absmax, fabsf(__uint_as_float(w[e] & 0xffff0000u)));
      }
    }
  }
  return absmax;
}

// Second pass: Q per-row quantise into TMEM (step a1); returns
// s_q * sm_scale * log2(e).
__device__ __forceinline__ float q_prologue(const AttnParams& p, const RowInfo& ri, float absmax, uint32_t tq) {
  const uint4* src = reinterpret_cast<const uint4*>(p.q + ri.off);
  float mul, s_q;
  if (p.q_mode == 1) {  // int8 grid, scale absmax/127, round half even
    mul = absmax > 0.f ? __fdiv_rn(127.f, absmax) : 0.f;
    s_q = __fdiv_rn(absmax, 127.f);
  } else {  // lossless fp16 container: power-of-two scale, absmax in [64, 128)
    const int k = absmax > 0.f ? imin(127, 133 - (int)((__float_as_uint(absmax) >> 23) & 0xff)) : 0;
    mul = __uint_as_float((uint32_t)(127 + k) << 23);
    s_q = __uint_as_float((uint32_t)(127 - k) << 23);
  }
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t pk[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 v = ri.valid ? __ldg(src + cc * 8 + k) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a = __uint_as_float(w[e] << 16) * mul;
        float b = __uint_as_float(w[e] & 0xffff0000u) * mul;
        if (p.q_mode == 1) {
          a = fminf(127.f, fmaxf(-127.f, rintf(a)));
          b = fminf(127.f, fmaxf(-127.f, rintf(b)));
        }
        pk[k * 4 + e] = pack_half2(a, b);
      }
    }
    tmem_st32(tq + cc * 32, pk);
  }
  return s_q * p.sm_scale_log2;
}

// out = O / l (x s_p on the u8 grid) -> bf16 (step a8).
__device__ __forceinline__ bool epilogue(const AttnParams& p, const Ctx& c, const RowInfo& ri, int k_unit,
                                         uint32_t to, const float* l_rows, const float* sp_rows, int r) {
  if (!c.warp_wait(B_OFULL, k_unit & 1, 41)) return false;
  if (!c.warp_wait(B_STATS + (k_unit & 1), (k_unit >> 1) & 1, 42)) return false;
  tc_fence_after();
  const float l = l_rows[(k_unit & 1) * 2 * kRows + r] + l_rows[(k_unit & 1) * 2 * kRows + kRows + r];
  const float sp = sp_rows[(k_unit & 1) * kRows + r];
  const float fin = l > 0.f ? (p.p_mode == 1 ? sp : 1.f) / l : 0.f;
  __nv_bfloat16* orow = p.out + ri.off;
#pragma unroll 1
  for (int cc = 0; cc < 8; ++cc) {
    uint32_t o[32];
    tmem_ld32(to + cc * 32, o);
    tmem_wait_ld(o);
    if (ri.valid) {
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        __nv_bfloat162 v =
            __floats2bfloat162_rn(__uint_as_float(o[2 * q]) * fin, __uint_as_float(o[2 * q + 1]) * fin);
        w[q] = *reinterpret_cast<uint32_t*>(&v);
      }
      uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
  }
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(c.bar(B_OEMPTY));
  return true;
}

__device__ __forceinline__ void role_correction(const AttnParams& p, const Ctx& c, uint8_t* sm) {
  const int r = threadIdx.x - 384;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  float* c_rows = reinterpret_cast<float*>(sm + kSmRows);
  const float* l_rows = c_rows + 2 * kRows;
  const float* sp_rows = c_rows + 6 * kRows;
  int k_unit = 0;
  bool ok = true;
  RowInfo prev{};
  for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++k_unit) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const RowInfo ri = row_info(p, un, sg, r);
    const float absmax = q_absmax(p, ri);
    // Q of this unit may replace the previous unit's once its last QK^T is done
    if (k_unit > 0 && !(ok = c.warp_wait(B_QEMPTY, (k_unit - 1) & 1, 40))) break;
    tc_fence_after();
    c_rows[(k_unit & 1) * kRows + r] = q_prologue(p, ri, absmax, c.tb + lane_off + kTmQ);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(B_QFULL));
    if (k_unit > 0) ok = epilogue(p, c, prev, k_unit - 1, c.tb + lane_off + kTmO, l_rows, sp_rows, r);
    prev = ri;
  }
  if (ok && k_unit > 0) (void)epilogue(p, c, prev, k_unit - 1, c.tb + lane_off + kTmO, l_rows, sp_rows, r);
  tmem_wait_st();
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ AttnMaps m) {
  extern __shared__ uint8_t smraw[];
  // 1024-byte aligned base by pointer arithmetic on the shared array, so the
  // compiler keeps every access through `sm` in the shared address space
  uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  Ctx c;
  c.sbase = smem_u32(sm);
  c.wc = WaitCtl{p.err, p.wait_ns};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kSmTmemSlot);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(c.bar(B_KFULL + s), 1);
      mbar_init(c.bar(B_KEMPTY + s), 8);  // every softmax warp, after reading the K scales
      mbar_init(c.bar(B_VFULL + s), 1);
      mbar_init(c.bar(B_VEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(B_SFULL + b), 1);
      mbar_init(c.bar(B_PFULL + b), 8);
    }
    mbar_init(c.bar(B_QFULL), 4);
    mbar_init(c.bar(B_QEMPTY), 1);
    mbar_init(c.bar(B_OFULL), 1);
    mbar_init(c.bar(B_OEMPTY), 4);
    mbar_init(c.bar(B_STATS), 8);
    mbar_init(c.bar(B_STATS + 1), 8);
    mbar_init(c.bar(B_STALL), 1);
    mbar_init(c.bar(B_DRAIN), 1);
    fence_mbar_init();
    tma_prefetch_map(&m.k);
    tma_prefetch_map(&m.v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  // scale slots start at zero: columns past a tile's width then hold finite
  // stale scales, which the softmax multiplies by p = 0
  for (int i = threadIdx.x; i < kSlots * 128; i += kThreads) reinterpret_cast<float*>(sm + kSmScale)[i] = 0.f;
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tb = *tmem_slot;

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) role_producer(p, m, c);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) role_mma(p, c);
  } else if (warp >= 4 && warp < 12) {
    role_softmax(p, c, sm);
  } else if (warp >= 12) {
    role_correction(p, c, sm);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(c.tb, 512);
  }
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, const AttnMaps& m, int n_sm, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
  if (e != cudaSuccess) return e;
  const int grid = imax(1, imin(p.n_units, n_sm));
  attention_kernel<<<grid, kThreads, kAttnSmem, st>>>(p, m);
  return cudaGetLastError();
}

}  // namespace pa
