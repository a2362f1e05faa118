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
//   warps 4-7     softmax, one query row per thread (TMEM lane = row)
//   warps 8-11    Q prologue of the next unit and epilogue of the previous one
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

constexpr int kThreads = 384;
constexpr int kSlots = 3;                              // depth of the K ring and of the V ring
constexpr int kKTileBytes = kTileKeys * kHeadDim * 2;  // 32 KB: 4 regions of 64 keys x 128 B
constexpr int kVTileBytes = kHeadDim * kTileKeys * 2;  // 32 KB: 256 dims x 128 B
// Shared memory, offsets from a 1024-byte aligned base.
constexpr int kSmK = 0;
constexpr int kSmV = kSmK + kSlots * kKTileBytes;
constexpr int kSmScale = kSmV + kSlots * kVTileBytes;  // per V slot: ks[64] then vs[64]
constexpr int kSmRows = kSmScale + kSlots * 512;       // c[2][128], l[2][128], sp[2][128] floats
constexpr int kSmBars = kSmRows + 3 * 2 * kRows * 4;
enum : int {
  B_KFULL = 0, B_KEMPTY = 3, B_VFULL = 6, B_VEMPTY = 9, B_SFULL = 12, B_PFULL = 14, B_PVDONE = 16,
  B_QFULL = 17, B_QEMPTY = 18, B_OFULL = 19, B_OEMPTY = 20, B_STATS = 21 /* two, by unit parity */,
  B_STALL = 23, B_DRAIN = 24, kNumBars = 25
};
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
  uint32_t kc = 0, vc = 0;
  int k_last[kSlots], v_last[kSlots];
  for (int s = 0; s < kSlots; ++s) k_last[s] = v_last[s] = -1;
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
        mbar_expect_tx(fb, kKTileBytes);
        const uint32_t dst = c.sbase + kSmK + s * kKTileBytes;
        for (int r = 0; r < 4; ++r) tma_load_3d(dst + r * 8192, &m.k, fb, r * 64, crow, un.g);
        k_last[s] = (int)ph;
        ++kc;
      }
      {
        const int s = vc % kSlots;
        const uint32_t ph = (vc / kSlots) & 1;
        if (!(ok = mbar_wait(c.bar(B_VEMPTY + s), ph ^ 1, c.wc, 11))) break;
        const uint32_t fb = c.bar(B_VFULL + s);
        const uint32_t sbytes = (uint32_t)(tg.nb * kPage * 4);
        mbar_expect_tx(fb, kVTileBytes + 2 * sbytes);
        tma_load_3d(c.sbase + kSmV + s * kVTileBytes, &m.v, fb, crow, 0, un.g);
        const size_t soff = (size_t)un.g * p.n_tok_cap + crow;
        bulk_load(c.sbase + kSmScale + s * 512, p.ks + soff, sbytes, fb);
        bulk_load(c.sbase + kSmScale + s * 512 + 256, p.vs + soff, sbytes, fb);
        v_last[s] = (int)ph;
        ++vc;
      }
    }
  }
  // every issued copy lands before the CTA may exit
  for (int s = 0; s < kSlots; ++s) {
    if (k_last[s] >= 0) (void)mbar_wait_drain(c.bar(B_KFULL + s), (uint32_t)k_last[s], kDrainNs);
    if (v_last[s] >= 0) (void)mbar_wait_drain(c.bar(B_VFULL + s), (uint32_t)v_last[s], kDrainNs);
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
#pragma unroll
        for (int s = 0; s < kHeadDim / 16; ++s)
          mma_ts(d, c.tb + kTmQ + 8 * s, sdesc_k_sw128(kaddr + (s >> 2) * 8192 + (s & 3) * 32), id, s > 0);
        mma_commit(c.bar(B_SFULL + (t & 1)));
        mma_commit(c.bar(B_KEMPTY + t % kSlots));
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
        for (int s = 0; s < tg.nb; ++s)
          mma_ts(c.tb + kTmO, a + 8 * s, sdesc_k_sw128(vaddr + 32 * s), id_pv, (jj > 0 || s > 0) ? 1u : 0u);
        mma_commit(c.bar(B_PVDONE));
        mma_commit(c.bar(B_VEMPTY + t % kSlots));
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
__device__ __forceinline__ void role_softmax(const AttnParams& p, const Ctx& c, uint8_t* sm) {
  const int r = threadIdx.x - 128;  // query row of this thread = TMEM lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  float* c_rows = reinterpret_cast<float*>(sm + kSmRows);
  float* l_rows = c_rows + 2 * kRows;
  float* sp_rows = c_rows + 4 * kRows;
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
    if (!(ok = c.warp_wait(B_QFULL, k_unit & 1, 30))) break;
    const float c_row = c_rows[(k_unit & 1) * kRows + r];
    float m_run = -INFINITY, l_run = 0.f, sp_prev = 1.f;
    for (int j = 0; j < n; ++j) {
      const uint32_t t = tc + j;
      const TileGeom tg = tile_geom(ug, j, p.S, p.W);
      if (!(ok = c.warp_wait(B_SFULL + (t & 1), (t >> 1) & 1, 31))) break;
      if (!(ok = c.warp_wait(B_VFULL + t % kSlots, (t / kSlots) & 1, 32))) break;
      tc_fence_after();
      const uint32_t sd = c.tb + lane_off + kTmS + (t & 1) * kTileKeys;
      uint32_t sa[32], sb[32];
      tmem_ld32(sd, sa);
      tmem_ld32(sd + 32, sb);
      tmem_wait_ld(sa);
      reg_fence(sb);
      const uint32_t sc = c.sbase + kSmScale + (t % kSlots) * 512;  // ks[64] then vs[64]
      const uint64_t vis = visible_columns(tg, t_row, p.S, p.W);
      const uint32_t vis_lo = (uint32_t)vis, vis_hi = (uint32_t)(vis >> 32);
      float x[64];
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int q4 = 0; q4 < 16; ++q4) {
        const float4 k4 = lds_f32x4(sc + 16 * q4);
        const float kq[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = 4 * q4 + e;
          const float sj = __uint_as_float(q < 32 ? sa[q] : sb[q - 32]);
          const bool on = ((q < 32 ? vis_lo : vis_hi) >> (q & 31)) & 1u;
          x[q] = on ? sj * kq[e] * c_row : -INFINITY;
          mx4[e] = fmaxf(mx4[e], x[q]);
        }
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      float alpha = 1.f;
      if (m_run == -INFINITY || mx > m_run + 8.f) {  // move the reference only when it grows by > 2^8
        const float mnew = fmaxf(m_run, mx);
        alpha = m_run == -INFINITY ? 0.f : ex2_approx(m_run - mnew);
        m_run = mnew;
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run + ev;
      float ps4[4] = {0.f, 0.f, 0.f, 0.f}, pm4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q4 = 0; q4 < 16; ++q4) {
        const float4 v4 = lds_f32x4(sc + 256 + 16 * q4);
        const float vq[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = 4 * q4 + e;
          const float pj = ex2_approx(x[q] - mref);
          ps4[e] += pj;
          const bool on = ((q < 32 ? vis_lo : vis_hi) >> (q & 31)) & 1u;
          x[q] = on ? pj * vq[e] : 0.f;  // V scale folded into P
          pm4[e] = fmaxf(pm4[e], x[q]);
        }
      }
      const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      const float pmax = fmaxf(fmaxf(pm4[0], pm4[1]), fmaxf(pm4[2], pm4[3]));
      l_run = l_run * alpha + psum;
      float corr = alpha;
      if (p.p_mode == 1) {  // P' per row on the u8 grid, scale max/255
        const float sp = pmax > 0.f ? __fdiv_rn(pmax, 255.f) : sp_prev;
        const float inv = pmax > 0.f ? __fdiv_rn(255.f, pmax) : 0.f;
#pragma unroll
        for (int q = 0; q < 64; ++q) x[q] = rintf(x[q] * inv);
        corr = alpha * __fdiv_rn(sp_prev, sp);
        sp_prev = sp;
      }
      uint32_t pk[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) pk[q] = pack_half2(x[2 * q], x[2 * q + 1]);
      tmem_st32(sd, pk);
      if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
        // O holds PV up to tile j-1 once that MMA is done; rescale it in place
        if (!(ok = c.warp_wait(B_PVDONE, (t - 1) & 1, 33))) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t o[32];
          tmem_ld32(c.tb + lane_off + kTmO + cc * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * corr);
          tmem_st32(c.tb + lane_off + kTmO + cc * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(B_PFULL + (t & 1)));
    }
    if (!ok) break;
    tc += n;
    l_rows[(k_unit & 1) * kRows + r] = l_run;
    sp_rows[(k_unit & 1) * kRows + r] = sp_prev;
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

// Q per-row quantise into TMEM (step a1); returns s_q * sm_scale * log2(e).
__device__ __forceinline__ float q_prologue(const AttnParams& p, const RowInfo& ri, uint32_t tq) {
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
  const float l = l_rows[(k_unit & 1) * kRows + r];
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
  const int r = threadIdx.x - 256;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  float* c_rows = reinterpret_cast<float*>(sm + kSmRows);
  const float* l_rows = c_rows + 2 * kRows;
  const float* sp_rows = c_rows + 4 * kRows;
  int k_unit = 0;
  bool ok = true;
  RowInfo prev{};
  for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++k_unit) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const RowInfo ri = row_info(p, un, sg, r);
    // Q of this unit may replace the previous unit's once its last QK^T is done
    if (k_unit > 0 && !(ok = c.warp_wait(B_QEMPTY, (k_unit - 1) & 1, 40))) break;
    tc_fence_after();
    c_rows[(k_unit & 1) * kRows + r] = q_prologue(p, ri, c.tb + lane_off + kTmQ);
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
      mbar_init(c.bar(B_KEMPTY + s), 1);
      mbar_init(c.bar(B_VFULL + s), 1);
      mbar_init(c.bar(B_VEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(B_SFULL + b), 1);
      mbar_init(c.bar(B_PFULL + b), 4);
    }
    mbar_init(c.bar(B_PVDONE), 1);
    mbar_init(c.bar(B_QFULL), 4);
    mbar_init(c.bar(B_QEMPTY), 1);
    mbar_init(c.bar(B_OFULL), 1);
    mbar_init(c.bar(B_OEMPTY), 4);
    mbar_init(c.bar(B_STATS), 4);
    mbar_init(c.bar(B_STATS + 1), 4);
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tb = *tmem_slot;

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) role_producer(p, m, c);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) role_mma(p, c);
  } else if (warp >= 4 && warp < 8) {
    role_softmax(p, c, sm);
  } else if (warp >= 8) {
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
