// Kernels of the windowed prefill attention over a paged int8 KV pool (sm_103a).
//
//   widen_kernel      page gather through the block table: int8 K/V pages ->
//                     contiguous integer-valued fp16 copies (K row-major, V
//                     transposed) plus per-token scales, visible blocks only.
//   attention_kernel  per 128-row work unit: Q per-row quantise into TMEM,
//                     then per 64-key tile: QK^T on tcgen05 (fp32 in TMEM),
//                     scale + mask + online softmax, V scale folded into P,
//                     P quantised into TMEM, PV on tcgen05 accumulating O in
//                     TMEM; epilogue O / l -> bf16.
//
// The method is the one of "int8 tensor-core prefill attention" (sections
// "Summary" and "Why the attention, and why tensor cores"): int8 K/V read from
// the paged pool, Q quantised per row, per-row Q, per-token K and softmax
// scales applied to the integer-valued scores, the per-token V scale folded
// into P before P is quantised per row, and masked blocks skipped.  sm_103a has
// no integer tcgen05 MMA, so the integer codes ride in fp16 containers on
// tcgen05.mma kind::f16 (exact: |code| <= 255 fits the 11-bit significand and
// the fp32 accumulator holds the integer sums exactly below 2^24).
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

// ======================================================================
// Widening (gather) pass
// ======================================================================
constexpr int kWidenThreads = 256;

__global__ void __launch_bounds__(kWidenThreads) widen_kernel(const WidenParams p) {
  __shared__ __align__(16) int8_t vpage[kPage * 8 * kHeadDim];  // up to 8 kv heads staged
  const int blk = blockIdx.x;
  const int tid = threadIdx.x;
  int s = 0;
  while (s + 1 < p.n_seq && p.seqs[s + 1].tok_off <= blk * kPage) ++s;
  const SeqGeom sg = p.seqs[s];
  const int b = blk - sg.tok_off / kPage;
  const int kb = stored_to_logical_block(sg, b);
  const int row0 = blk * kPage;
  const int phys = p.block_table[(size_t)sg.bt_row * p.bt_stride + kb];
  const bool bad = phys < 0 || phys >= p.n_pool;
  if (bad && tid == 0) atomicCAS(p.err, 0, DEV_ERR_BAD_PAGE);
  const int n_valid = bad ? 0 : imax(0, imin(kPage, sg.n_ctx - kb * kPage));
  const int HKV = p.HKV;
  const size_t page_base = (size_t)(bad ? 0 : phys) * kPage * HKV * kHeadDim;

  // K: 16-byte chunks of 16 codes, (token, head, chunk) over the block.
  for (int idx = tid; idx < kPage * HKV * 16; idx += kWidenThreads) {
    const int c = idx & 15;
    const int g = (idx >> 4) % HKV;
    const int tk = (idx >> 4) / HKV;
    int4 raw = make_int4(0, 0, 0, 0);
    if (tk < n_valid)
      raw = *reinterpret_cast<const int4*>(p.k_pool + page_base + ((size_t)tk * HKV + g) * kHeadDim + c * 16);
    const int8_t* cb = reinterpret_cast<const int8_t*>(&raw);
    __align__(16) __half h[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) h[e] = __int2half_rn((int)cb[e]);
    int4* dst = reinterpret_cast<int4*>(p.kw + ((size_t)g * p.n_tok_cap + row0 + tk) * kHeadDim + c * 16);
    dst[0] = reinterpret_cast<const int4*>(h)[0];
    dst[1] = reinterpret_cast<const int4*>(h)[1];
  }
  // V: stage the page, then write each (head, dim) column of 16 tokens.
  for (int idx = tid; idx < kPage * HKV * 16; idx += kWidenThreads) {
    const int tk = idx / (HKV * 16);
    int4 raw = make_int4(0, 0, 0, 0);
    if (tk < n_valid) raw = *reinterpret_cast<const int4*>(p.v_pool + page_base + (size_t)idx * 16);
    reinterpret_cast<int4*>(vpage)[idx] = raw;
  }
  __syncthreads();
  for (int col = tid; col < HKV * kHeadDim; col += kWidenThreads) {
    const int g = col / kHeadDim, d = col % kHeadDim;
    __align__(16) __half h[16];
#pragma unroll
    for (int tk = 0; tk < kPage; ++tk) h[tk] = __int2half_rn((int)vpage[(tk * HKV + g) * kHeadDim + d]);
    int4* dst = reinterpret_cast<int4*>(p.vt + ((size_t)g * kHeadDim + d) * p.n_tok_cap + row0);
    dst[0] = reinterpret_cast<const int4*>(h)[0];
    dst[1] = reinterpret_cast<const int4*>(h)[1];
  }
  // Scales (0 past the end of the context) and the running max of V scales.
  if (tid < kPage * HKV) {
    const int tk = tid / HKV, g = tid % HKV;
    float ksv = 0.f, vsv = 0.f;
    if (tk < n_valid) {
      const size_t slot = ((size_t)phys * kPage + tk) * HKV + g;
      ksv = p.k_scale[slot];
      vsv = p.v_scale[slot];
    }
    p.ks[(size_t)g * p.n_tok_cap + row0 + tk] = ksv;
    p.vs[(size_t)g * p.n_tok_cap + row0 + tk] = vsv;
    if (vsv > 0.f) atomicMax(p.vsmax + s * HKV + g, __float_as_uint(vsv));
  }
}

cudaError_t launch_widen(const WidenParams& p, cudaStream_t st) {
  if (p.HKV > 8) return cudaErrorInvalidValue;
  widen_kernel<<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p);
  return cudaGetLastError();
}

// ======================================================================
// Attention kernel
// ======================================================================
constexpr int kAttnThreads = 128;
// Shared memory (offsets from a 1024-byte aligned base).
constexpr int kSmQ = 0;                          // Q bf16: 4 regions of 128 rows x 128 B (64 KB)
constexpr int kSmStage0 = 65536;                 // stage s: K (4 x 64 rows x 128 B) then Vt (256 x 128 B)
constexpr int kStageBytes = 65536;
constexpr int kSmKOff = 0, kSmVOff = 32768;
constexpr int kSmScales = kSmStage0 + 2 * kStageBytes;  // stage s: ks[64] at +s*512, vs[64] at +s*512+256
constexpr int kAttnSmem = kSmScales + 1024 + 1024;     // + alignment slack
// TMEM columns.
constexpr uint32_t kTmO = 0;     // O accumulator 128 x 256 fp32
constexpr uint32_t kTmQ = 256;   // Q (fp16 pairs) 128 x 128 columns
constexpr uint32_t kTmS = 384;   // S 128 x 64 fp32; P (fp16 pairs) aliases its first 32 columns

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Power-of-two exponent e with 2^(e-1) <= x < 2^e, clamped to [-100, 100];
// 0 for x <= 0.
__device__ __forceinline__ int pow2_ceil_exp(float x) {
  if (!(x > 0.f)) return 0;
  const int eb = (int)((__float_as_uint(x) >> 23) & 0xff);
  int e = eb - 126;  // x in [2^(eb-127), 2^(eb-126))
  return imax(-100, imin(100, e));
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ AttnMaps m) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[5];  // 0: Q, 1-2: K/V stages, 3: MMA, 4: never armed (test hook)
  __shared__ uint32_t tmem_base_s;

  const int tid = threadIdx.x, warp = tid >> 5;
  const WaitCtl wc{p.err, p.wait_ns};
  const uint32_t bar_q = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[3]);
  const uint32_t bar_kv0 = smem_u32(&bars[1]);
  const uint32_t sm_base = smem_u32(sm);

  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
    tma_prefetch_map(&m.q);
    tma_prefetch_map(&m.k);
    tma_prefetch_map(&m.v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_s), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_s;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  const Unit un = p.units[blockIdx.x];
  const SeqGeom sg = p.seqs[un.seq];
  const UnitGeom ug = unit_geom(un.t0, p.TQ, sg, p.S, p.W);
  const int n_tiles = ug.n_tiles;

  auto issue_tile = [&](int i) {
    const int st = i & 1;
    const TileGeom tg = tile_geom(ug, i, p.S, p.W);
    const int crow = logical_block_row(sg, tg.kb0);
    const uint32_t bar = bar_kv0 + 8 * st;
    const uint32_t kbase = sm_base + kSmStage0 + st * kStageBytes + kSmKOff;
    const uint32_t vbase = sm_base + kSmStage0 + st * kStageBytes + kSmVOff;
    const uint32_t sbase = sm_base + kSmScales + st * 512;
    const uint32_t sbytes = static_cast<uint32_t>(tg.nb * kPage * 4);
    mbar_expect_tx(bar, 32768u + 32768u + 2u * sbytes);
    for (int c = 0; c < 4; ++c) tma_load_3d(kbase + c * 8192, &m.k, bar, c * 64, crow, un.g);
    tma_load_3d(vbase, &m.v, bar, crow, 0, un.g);
    const size_t soff = (size_t)un.g * p.n_tok_cap + crow;
    bulk_load(sbase, p.ks + soff, sbytes, bar);
    bulk_load(sbase + 256, p.vs + soff, sbytes, bar);
  };

  int issued = 0;  // tiles whose loads were issued (tracked by thread 0)
  if (tid == 0) {
    mbar_expect_tx(bar_q, 65536u);
    const int qrow = sg.q_off + (un.t0 - sg.q_start);
    for (int c = 0; c < 4; ++c) tma_load_3d(sm_base + kSmQ + c * 16384, &m.q, bar_q, c * 64, un.g * p.G, qrow);
    for (; issued < 2 && issued < n_tiles; ++issued) issue_tile(issued);
  }

  // ---- prologue: Q per-row quantise into TMEM (row r = tid)
  const int r = tid;
  const int t_row = un.t0 + r / p.G;
  const int h_row = un.g * p.G + r % p.G;
  bool ok = mbar_wait(p.debug_stall ? smem_u32(&bars[4]) : bar_q, 0, wc, 1);
  const bool q_landed = ok && !p.debug_stall;
  float c_row = 0.f;  // s_q * sm_scale * log2(e)
  if (ok) {
    const uint8_t* qs = sm + kSmQ;
    float absmax = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = *reinterpret_cast<const uint4*>(qs + c * 16384 + r * 128 + ((k ^ (r & 7)) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          absmax = fmaxf(absmax, fabsf(__uint_as_float(w[e] << 16)));
          absmax = fmaxf(absmax, fabsf(__uint_as_float(w[e] & 0xffff0000u)));
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
    c_row = s_q * p.sm_scale_log2;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = *reinterpret_cast<const uint4*>(qs + c * 16384 + r * 128 + ((k ^ (r & 7)) << 4));
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
      tmem_st32(tb + lane_off + kTmQ + c * 32, pk);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  ok = __syncthreads_and(ok);
  tc_fence_after();

  // V-scale normaliser: P' = p * s_v * 2^-ev stays below 256.
  const float ev = (float)pow2_ceil_exp(__uint_as_float(p.vsmax[un.seq * p.HKV + un.g]));
  const int lo_row = p.W > 0 ? imax(0, t_row / kPage + 1 - p.W) : 0;
  float m_run = -INFINITY, l_run = 0.f, sp_prev = 1.f;
  uint32_t mma_phase = 0;
  bool mma_pending = false;
  int consumed = 0;  // tiles whose K/V wait completed

  for (int i = 0; i < n_tiles && ok; ++i) {
    const int st = i & 1;
    const TileGeom tg = tile_geom(ug, i, p.S, p.W);
    const int kw = tg.nb * kPage;
    const int key0 = tg.kb0 * kPage;
    ok = mbar_wait(bar_kv0 + 8 * st, (i >> 1) & 1, wc, 2);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    consumed = i + 1;
    // ---- S = Q K^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kbase = sm_base + kSmStage0 + st * kStageBytes + kSmKOff;
      const uint32_t id = idesc_f16(128, kw, false, false);
#pragma unroll
      for (int s = 0; s < 16; ++s)
        mma_ts(tb + kTmS, tb + kTmQ + 8 * s, sdesc_k_sw128(kbase + (s >> 2) * 8192 + (s & 3) * 32), id, s > 0);
      mma_commit(bar_mma);
      mma_pending = true;
    }
    ok = mbar_wait(bar_mma, mma_phase, wc, 3);
    mma_phase ^= 1;
    if (tid == 0) mma_pending = !ok;
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (!ok) break;

    uint32_t sa[32], sb[32];
    tmem_ld32(tb + lane_off + kTmS, sa);
    tmem_ld32(tb + lane_off + kTmS + 32, sb);
    tmem_wait_ld(sa);
    reg_fence(sb);

    // ---- scale, mask, online softmax (this thread owns row r)
    const float* ksm = reinterpret_cast<const float*>(sm + kSmScales + st * 512);
    const float* vsm = ksm + 64;
    float x[64];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const float sj = __uint_as_float(j < 32 ? sa[j] : sb[j - 32]);
      const int key = key0 + j;
      bool vis = j < kw;
      if (tg.needs_mask)
        vis = vis && key <= t_row && (p.W <= 0 || key / kPage < p.S || key / kPage >= lo_row);
      x[j] = vis ? sj * ksm[j] * c_row : -INFINITY;
      mx = fmaxf(mx, x[j]);
    }
    float alpha = 1.f;
    if (m_run == -INFINITY || mx > m_run + 8.f) {
      const float mnew = fmaxf(m_run, mx);
      alpha = m_run == -INFINITY ? 0.f : ex2_approx(m_run - mnew);
      m_run = mnew;
    }
    const float mref = m_run == -INFINITY ? 0.f : m_run + ev;
    float psum = 0.f, pmax = 0.f;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const float pj = ex2_approx(x[j] - mref);
      psum += pj;
      x[j] = j < kw ? pj * vsm[j] : 0.f;  // V scale folded into P
      pmax = fmaxf(pmax, x[j]);
    }
    l_run = l_run * alpha + psum;
    float corr = alpha;
    if (p.p_mode == 1) {  // P' per row on the u8 grid, scale max/255
      const float sp = pmax > 0.f ? __fdiv_rn(pmax, 255.f) : sp_prev;
      const float inv = pmax > 0.f ? __fdiv_rn(255.f, pmax) : 0.f;
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = rintf(x[j] * inv);
      corr = alpha * __fdiv_rn(sp_prev, sp);
      sp_prev = sp;
    }
    uint32_t pk[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) pk[j] = pack_half2(x[2 * j], x[2 * j + 1]);
    tmem_st32(tb + lane_off + kTmS, pk);
    // ---- rescale O when this warp has a row whose reference moved
    if (i > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        tmem_ld32(tb + lane_off + kTmO + c * 32, o);
        tmem_wait_ld(o);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * corr);
        tmem_st32(tb + lane_off + kTmO + c * 32, o);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    // ---- O (+)= P V
    if (tid == 0) {
      tc_fence_after();
      const uint32_t vbase = sm_base + kSmStage0 + st * kStageBytes + kSmVOff;
      const uint32_t id = idesc_f16(128, 256, false, false);
      for (int s = 0; s < tg.nb; ++s)
        mma_ts(tb + kTmO, tb + kTmS + 8 * s, sdesc_k_sw128(vbase + s * 32), id, (i > 0 || s > 0) ? 1u : 0u);
      mma_commit(bar_mma);
      mma_pending = true;
    }
    ok = mbar_wait(bar_mma, mma_phase, wc, 4);
    mma_phase ^= 1;
    if (tid == 0) mma_pending = !ok;
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (ok && tid == 0 && issued < n_tiles && issued == i + 2) {
      issue_tile(issued);
      ++issued;
    }
  }

  // ---- epilogue: out = O / l (x s_p on the u8 grid) -> bf16
  ok = __syncthreads_and(ok);
  if (ok) {
    const float fin = l_run > 0.f ? (p.p_mode == 1 ? sp_prev : 1.f) / l_run : 0.f;
    const bool valid = t_row >= sg.q_start && t_row < sg.q_start + sg.n_q;
    __nv_bfloat16* orow = p.out + ((size_t)(sg.q_off + t_row - sg.q_start) * p.HQ + h_row) * kHeadDim;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t o[32];
      tmem_ld32(tb + lane_off + kTmO + c * 32, o);
      tmem_wait_ld(o);
      if (valid) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(o[2 * j]) * fin,
                                                   __uint_as_float(o[2 * j + 1]) * fin);
          w[j] = *reinterpret_cast<uint32_t*>(&v);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      }
    }
  }

  // ---- teardown: never leave copies or MMAs in flight, then free TMEM
  if (tid == 0) {
    const uint64_t drain_ns = 200000000ull;
    if (mma_pending) (void)mbar_wait_drain(bar_mma, mma_phase, drain_ns);
    // loads issued but not consumed: tiles [consumed, issued); each stage has
    // at most one such load, whose phase is the stage's current one
    for (int i = consumed; i < issued; ++i) (void)mbar_wait_drain(bar_kv0 + 8 * (i & 1), (i >> 1) & 1, drain_ns);
    if (!q_landed) (void)mbar_wait_drain(bar_q, 0, drain_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t launch_attention(const AttnParams& p, const AttnMaps& m, int n_sm, cudaStream_t st) {
  (void)n_sm;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attention_kernel<<<p.n_units, kAttnThreads, kAttnSmem, st>>>(p, m);
  return cudaGetLastError();
}

// ======================================================================
// Debug exports (tests only): the same geometry helpers as the kernels.
// ======================================================================
__global__ void debug_gather_kernel(const WidenParams p, int seq, int8_t* k_out, int8_t* v_out, float* ks_out,
                                    float* vs_out, int32_t* tok_out) {
  const SeqGeom sg = p.seqs[seq];
  const int n_rows = sg.n_blocks * kPage;
  for (int rr = blockIdx.x; rr < n_rows; rr += gridDim.x) {
    const int kb = stored_to_logical_block(sg, rr / kPage);
    const int tok = kb * kPage + rr % kPage;
    const int row = sg.tok_off + rr;
    if (threadIdx.x == 0) tok_out[rr] = tok < sg.n_ctx ? tok : -1;
    for (int gd = threadIdx.x; gd < p.HKV * kHeadDim; gd += blockDim.x) {
      const int g = gd / kHeadDim, d = gd % kHeadDim;
      k_out[((size_t)g * n_rows + rr) * kHeadDim + d] =
          (int8_t)__half2int_rn(p.kw[((size_t)g * p.n_tok_cap + row) * kHeadDim + d]);
      v_out[((size_t)g * n_rows + rr) * kHeadDim + d] =
          (int8_t)__half2int_rn(p.vt[((size_t)g * kHeadDim + d) * p.n_tok_cap + row]);
    }
    if (threadIdx.x < p.HKV) {
      const int g = threadIdx.x;
      ks_out[(size_t)g * n_rows + rr] = p.ks[(size_t)g * p.n_tok_cap + row];
      vs_out[(size_t)g * n_rows + rr] = p.vs[(size_t)g * p.n_tok_cap + row];
    }
  }
}

cudaError_t launch_debug_gather(const WidenParams& p, int seq, int8_t* k_out, int8_t* v_out, float* ks_out,
                                float* vs_out, int32_t* tok_out, cudaStream_t st) {
  debug_gather_kernel<<<256, 256, 0, st>>>(p, seq, k_out, v_out, ks_out, vs_out, tok_out);
  return cudaGetLastError();
}

// Per unit: the key blocks its tiles visit (in visiting order, -1 padded) and,
// per row, how many keys the kernel's mask lets through.
__global__ void debug_maskset_kernel(const SeqGeom* seqs, const Unit* units, int TQ, int G, int S, int W,
                                     int32_t* row_counts, int32_t* unit_blocks, int cap) {
  const Unit un = units[blockIdx.x];
  const SeqGeom sg = seqs[un.seq];
  const UnitGeom ug = unit_geom(un.t0, TQ, sg, S, W);
  const int r = threadIdx.x;
  const int t_row = un.t0 + r / G;
  int count = 0, nblk = 0;
  for (int i = 0; i < ug.n_tiles; ++i) {
    const TileGeom tg = tile_geom(ug, i, S, W);
    if (r == 0)
      for (int b = 0; b < tg.nb; ++b) {
        if (nblk < cap) unit_blocks[(size_t)blockIdx.x * cap + nblk] = tg.kb0 + b;
        ++nblk;
      }
    if (!tg.needs_mask) {
      count += tg.nb * kPage;
    } else {
      for (int j = tg.kb0 * kPage; j < (tg.kb0 + tg.nb) * kPage; ++j) count += key_visible(t_row, j, S, W) ? 1 : 0;
    }
  }
  if (r == 0)
    for (int k = nblk; k < cap; ++k) unit_blocks[(size_t)blockIdx.x * cap + k] = -1;
  row_counts[(size_t)blockIdx.x * kRows + r] = count;
}

cudaError_t launch_debug_maskset(const SeqGeom* seqs, const Unit* units, int n_units, int TQ, int G, int S, int W,
                                 int32_t* row_counts, int32_t* unit_blocks, int cap, cudaStream_t st) {
  debug_maskset_kernel<<<n_units, kRows, 0, st>>>(seqs, units, TQ, G, S, W, row_counts, unit_blocks, cap);
  return cudaGetLastError();
}

}  // namespace pa
