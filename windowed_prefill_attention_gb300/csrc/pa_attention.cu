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
constexpr int kSmStage = kSmXchg + 8 * kRows * 4;      // correction warps: 4 x [32 rows][128 B]
constexpr int kSmBars = kSmStage + 4 * 4096;
enum : int {
  B_KFULL = 0, B_KEMPTY = 3, B_VFULL = 6, B_VEMPTY = 9, B_SFULL = 12, B_PFULL = 14,
  B_QFULL = 16, B_QEMPTY = 17, B_OFULL = 18, B_OEMPTY = 19, B_STATS = 20 /* two, by unit parity */,
  B_STALL = 22, B_DRAIN = 23, B_QSOON = 24, kNumBars = 25
};
// The MMA issuer arrives on B_QSOON when it issues QK^T for the tile kQSoon
// tiles before its unit's last; the correction warps then start loading the
// next unit's Q rows, so that they are in L2 when the unit's Q may be stored.
constexpr int kQSoon = 6;
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
    // Operands of the next QK^T.  They are prepared (K slot waited for,
    // descriptors built) right after the previous QK^T is issued, so that
    // PV(j-1) is followed at once by QK^T(j+1).
    uint32_t qk_d = 0, qk_id = 0;
    uint64_t qk_kd0 = 0;
    auto prep_qk = [&](int j) -> bool {
      const uint32_t t = tc + j;
      const uint32_t slot = t % kSlots;
      if (!mbar_wait(c.bar(B_KFULL + slot), (t / kSlots) & 1, c.wc, 21)) return false;
      qk_d = c.tb + kTmS + (t & 1) * kTileKeys;
      qk_id = idesc_f16(kRows, tile_width(ug, j) * kPage, true, true);  // bf16 Q, bf16 K codes
      qk_kd0 = sdesc_k_sw128(c.sbase + kSmK + slot * kKTileBytes);
      return true;
    };
    if (!(ok = prep_qk(0))) break;
    for (int j = 0; j <= n; ++j) {
      if (j < n) {  // S(j) = Q K(j)^T
        const uint32_t t = tc + j;
        tc_fence_after();
        // k-step s reads K bytes at (s/4)*8192 + (s%4)*32 from the slot: only
        // the descriptor's start-address field (address >> 4) moves
#pragma unroll
        for (int s = 0; s < kHeadDim / 16; ++s)
          mma_ts(qk_d, c.tb + kTmQ + 8 * s, qk_kd0 + (uint64_t)(((s >> 2) * 8192 + (s & 3) * 32) >> 4), qk_id, s > 0);
        mma_commit(c.bar(B_SFULL + (t & 1)));  // also frees K slot t: the softmax passes it on
        if (j == n - 1) mma_commit(c.bar(B_QEMPTY));
        if (j == imax(0, n - kQSoon)) mbar_arrive(c.bar(B_QSOON));
        if (j + 1 < n && !(ok = prep_qk(j + 1))) break;
      }
      if (j >= 1) {  // O (+)= P(j-1) V(j-1)
        const int jj = j - 1;
        const uint32_t t = tc + jj;
        // V(t) has landed: every softmax warp waited for its barrier (for the
        // V scales) before releasing P(t)
        if (!(ok = mbar_wait(c.bar(B_PFULL + (t & 1)), (t >> 1) & 1, c.wc, 22))) break;
        if (jj == 0 && k_unit > 0 && !(ok = mbar_wait(c.bar(B_OEMPTY), (k_unit - 1) & 1, c.wc, 24))) break;
        tc_fence_after();
        const uint32_t slot = t % kSlots;
        const uint32_t a = c.tb + kTmS + (t & 1) * kTileKeys;
        const uint64_t vd0 = sdesc_k_sw128(c.sbase + kSmV + slot * kVTileBytes);
        const int nb = tile_width(ug, jj);
        for (int s = 0; s < nb; ++s)
          mma_ts(c.tb + kTmO, a + 8 * s, vd0 + (uint64_t)(2 * s), id_pv, (jj > 0 || s > 0) ? 1u : 0u);
        mma_commit(c.bar(B_VEMPTY + slot));  // V slot t free; O holds PV up to tile t
        if (jj == n - 1) mma_commit(c.bar(B_OFULL));
      }
    }
    if (!ok) break;
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
      // this half's K scales (32 floats); its V scales follow 256 bytes later
      const float4* ks4 = reinterpret_cast<const float4*>(sm + kSmScale + (t % kSlots) * 512 + 128 * h);
      const float4* vs4 = ks4 + 16;
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
            const float4 k4 = ks4[q4];
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
            const float4 k4 = ks4[q4];
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
        const float4 v4 = vs4[q4];
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
  bool valid;
  size_t off;  // element offset of the row in q / out
};

__device__ __forceinline__ RowInfo row_info(const AttnParams& p, const Unit& un, const SeqGeom& sg, int r) {
  RowInfo ri;
  const int t_row = un.t0 + r / p.G;
  const int h_row = un.g * p.G + r % p.G;
  ri.valid = t_row >= sg.q_start && t_row < sg.q_start + sg.n_q;
  ri.off = ri.valid ? ((size_t)(sg.q_off + t_row - sg.q_start) * p.HQ + h_row) * kHeadDim : 0;
  return ri;
}

// Row-major global traffic of the correction warps goes through shared
// memory, 32 rows x 128 bytes per warp, so that one warp instruction moves
// four whole 128-byte lines (lane l: row 4k + l/8, 16-byte piece l%8) while
// the TMEM side keeps one row per thread.  Piece p of row i is kept at piece
// p ^ (i & 7), which makes both access patterns free of bank conflicts.
__device__ __forceinline__ uint4* stage_at(uint8_t* stage, int row, int piece) {
  return reinterpret_cast<uint4*>(stage + row * 128 + ((piece ^ (row & 7)) << 4));
}

// The rows lane `lane` moves in the four-rows-per-instruction pattern:
// row 4k + lane/8 of the warp's 32, k = 0..7.
struct LaneRows {
  uint32_t row[8];  // row index in q / out (element offset row * 256)
  uint32_t valid;   // bit k: row k is a query row of the call
};
__device__ __forceinline__ LaneRows lane_rows(const AttnParams& p, const Unit& un, const SeqGeom& sg, int qd,
                                              int lane) {
  LaneRows lr;
  lr.valid = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const RowInfo ri = row_info(p, un, sg, 32 * qd + 4 * k + (lane >> 3));
    lr.row[k] = (uint32_t)(ri.off / kHeadDim);
    lr.valid |= (ri.valid ? 1u : 0u) << k;
  }
  return lr;
}

// The row's absolute maximum, for the int8 grid only.
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

// Eight bf16 values -> their int8-grid codes rint(x * mul) clamped to
// [-127, 127], as bf16 (exact), same positions.
__device__ __forceinline__ uint4 quantise8(uint4 v, float mul) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = fminf(127.f, fmaxf(-127.f, rintf(__uint_as_float(w[e] << 16) * mul)));
    const float b = fminf(127.f, fmaxf(-127.f, rintf(__uint_as_float(w[e] & 0xffff0000u) * mul)));
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    w[e] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Q per-row quantise into TMEM (step a1); returns s_q * sm_scale * log2(e).
// PA_Q_BF16: Q's bf16 bits go to TMEM unchanged, s_q = 1.  PA_Q_INT8: codes
// on the pages' grid, s_q = absmax / 127.  64 columns of every row per round;
// the loads of the next round are in flight while one round is stored.
template <bool kInt8>
__device__ __forceinline__ float q_prologue(const AttnParams& p, const LaneRows& lr, float absmax, uint8_t* stage,
                                            uint32_t tq, int lane) {
  float s_q = 1.f, mul = 1.f;
  if (kInt8) {
    mul = absmax > 0.f ? __fdiv_rn(127.f, absmax) : 0.f;
    s_q = __fdiv_rn(absmax, 127.f);
  }
  float mk[8];  // the scale of each row this lane loads
  if (kInt8) {
#pragma unroll
    for (int k = 0; k < 8; ++k) mk[k] = __shfl_sync(0xffffffffu, mul, 4 * k + (lane >> 3));
  }
  const int pc = lane & 7;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  uint4 v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    v[k] = (lr.valid >> k) & 1u ? __ldg(reinterpret_cast<const uint4*>(p.q + (size_t)lr.row[k] * kHeadDim) + pc) : zero;
#pragma unroll
  for (int cb = 0; cb < 4; ++cb) {
    uint4 vn[8];
    if (cb < 3) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        vn[k] = (lr.valid >> k) & 1u
                    ? __ldg(reinterpret_cast<const uint4*>(p.q + (size_t)lr.row[k] * kHeadDim + (cb + 1) * 64) + pc)
                    : zero;
    }
    if (kInt8) {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = quantise8(v[k], mk[k]);
    }
    __syncwarp();  // the previous round's reads of the stage are done
#pragma unroll
    for (int k = 0; k < 8; ++k) *stage_at(stage, 4 * k + (lane >> 3), pc) = v[k];
    __syncwarp();
    uint32_t pk[32];
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) {
      const uint4 u = *stage_at(stage, lane, pp);
      pk[4 * pp] = u.x;
      pk[4 * pp + 1] = u.y;
      pk[4 * pp + 2] = u.z;
      pk[4 * pp + 3] = u.w;
    }
    tmem_st32(tq + cb * 32, pk);
    if (cb < 3) {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = vn[k];
    }
  }
  return s_q * p.sm_scale_log2;
}

// out = O / l (x s_p on the u8 grid) -> bf16 (step a8), 64 columns per round.
// O may be overwritten once the last round's TMEM loads are done, so the
// MMA issuer is released before the last stores.
__device__ __forceinline__ bool epilogue(const AttnParams& p, const Ctx& c, const LaneRows& lr, int k_unit,
                                         uint32_t to, const float* l_rows, const float* sp_rows, int r,
                                         uint8_t* stage, int lane) {
  if (!c.warp_wait(B_OFULL, k_unit & 1, 41)) return false;
  if (!c.warp_wait(B_STATS + (k_unit & 1), (k_unit >> 1) & 1, 42)) return false;
  tc_fence_after();
  const float l = l_rows[(k_unit & 1) * 2 * kRows + r] + l_rows[(k_unit & 1) * 2 * kRows + kRows + r];
  const float sp = sp_rows[(k_unit & 1) * kRows + r];
  const float fin = l > 0.f ? (p.p_mode == 1 ? sp : 1.f) / l : 0.f;
  const int pc = lane & 7;
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    uint32_t o0[32], o1[32];
    tmem_ld32(to + cb * 64, o0);
    tmem_ld32(to + cb * 64 + 32, o1);
    tmem_wait_ld(o0);
    reg_fence(o1);
    if (cb == 3) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(B_OEMPTY));
    }
    uint32_t w[32];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      __nv_bfloat162 a = __floats2bfloat162_rn(__uint_as_float(o0[2 * q]) * fin, __uint_as_float(o0[2 * q + 1]) * fin);
      __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(o1[2 * q]) * fin, __uint_as_float(o1[2 * q + 1]) * fin);
      w[q] = *reinterpret_cast<uint32_t*>(&a);
      w[16 + q] = *reinterpret_cast<uint32_t*>(&b);
    }
    __syncwarp();  // the previous round's reads of the stage are done
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) *stage_at(stage, lane, pp) = make_uint4(w[4 * pp], w[4 * pp + 1], w[4 * pp + 2], w[4 * pp + 3]);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if ((lr.valid >> k) & 1u)
        *(reinterpret_cast<uint4*>(p.out + (size_t)lr.row[k] * kHeadDim + cb * 64) + pc) =
            *stage_at(stage, 4 * k + (lane >> 3), pc);
  }
  return true;
}

__device__ __forceinline__ void role_correction(const AttnParams& p, const Ctx& c, uint8_t* sm) {
  const int r = threadIdx.x - 384;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3;
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  uint8_t* stage = sm + kSmStage + qd * 4096;
  float* c_rows = reinterpret_cast<float*>(sm + kSmRows);
  const float* l_rows = c_rows + 2 * kRows;
  const float* sp_rows = c_rows + 6 * kRows;
  int k_unit = 0;
  bool ok = true;
  Unit prev_un{};
  SeqGeom prev_sg{};
  for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++k_unit) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const RowInfo ri = row_info(p, un, sg, r);
    // fetch this unit's Q rows only when the previous unit is close to its
    // end: fetched earlier, they would be evicted from L2 before use
    if (k_unit > 0 && !(ok = c.warp_wait(B_QSOON, (k_unit - 1) & 1, 43))) break;
    if (ri.valid) bulk_prefetch_l2(p.q + ri.off, kHeadDim * 2);
    const float absmax = p.q_mode == 1 ? q_absmax(p, ri) : 0.f;
    const LaneRows lr = lane_rows(p, un, sg, qd, lane);
    // Q of this unit may replace the previous unit's once its last QK^T is done
    if (k_unit > 0 && !(ok = c.warp_wait(B_QEMPTY, (k_unit - 1) & 1, 40))) break;
    tc_fence_after();
    const uint32_t tq = c.tb + lane_off + kTmQ;
    c_rows[(k_unit & 1) * kRows + r] =
        p.q_mode == 1 ? q_prologue<true>(p, lr, absmax, stage, tq, lane) : q_prologue<false>(p, lr, absmax, stage, tq, lane);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(B_QFULL));
    if (k_unit > 0)
      ok = epilogue(p, c, lane_rows(p, prev_un, prev_sg, qd, lane), k_unit - 1, c.tb + lane_off + kTmO, l_rows,
                    sp_rows, r, stage, lane);
    prev_un = un;
    prev_sg = sg;
  }
  if (ok && k_unit > 0)
    (void)epilogue(p, c, lane_rows(p, prev_un, prev_sg, qd, lane), k_unit - 1, c.tb + lane_off + kTmO, l_rows,
                   sp_rows, r, stage, lane);
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
    mbar_init(c.bar(B_QSOON), 1);
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
