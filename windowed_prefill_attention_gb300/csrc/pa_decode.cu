// Split-KV flash decode over the paged int8 KV pool (sm_103a): one new query
// token per sequence attends to its visible keys under the same causal +
// sink/window block mask as the prefill ("int8 tensor-core prefill
// attention", section "Why the attention, and why tensor cores": the decode
// path keeps the prefill's window selection; section "Relation to open PRs":
// the int8 GQA flash-decode with KV splits whose Q-per-row / fold-V-into-P
// pattern the prefill follows).
//
// Decode reads every visible K/V code once and does 2 x G x 256 flops per
// code (G = q heads per kv head, <= 8): it is bound by HBM, not the tensor
// core.  So the int8 pool is read directly (no widening pass), a CTA takes 64
// blocks (1024 keys) of one (sequence, kv head), and the small products run
// on warp-level MMAs (mma.sync m16n8k16, fp16 containers, fp32 accumulate) in
// the transposed orientation, S^T = K Q^T and O^T = V^T P^T, so that keys and
// head dims fill M = 16 and the G query rows fill N = 8 with no padding.  In
// both the thread holds rows 2t, 2t+1 (t = lane % 4): the online-softmax state
// stays in registers.  Codes become exact fp16 pairs with one byte permute and
// one subtraction; the query enters as fp16 through a per-row power-of-two
// scale (lossless for bf16 input); P' = p * v_scale is normalised by the
// largest V scale the warp has met so far (a running power of two, rescaled
// like the running max) so that it stays in fp16's normal range.
//
// decode_split_kernel   one CTA per (sequence, kv head, split): 4 warps take
//                       the split's blocks in turn (two cp.async stages per
//                       warp), then combine in shared memory into one partial
//                       (row max, row sum, unnormalised O) per q head
// decode_combine_kernel one CTA per (sequence, q head): merges the splits'
//                       partials and writes bf16
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kDecWarps = 4;
constexpr int kRowPitch = 272;                       // staged code row: 256 B + 16 (bank spread, 16-B aligned)
constexpr int kStagePage = kPage * kRowPitch;        // 4352
constexpr int kStageBuf = 2 * kStagePage + 128;      // K page, V page, 16 K + 16 V scales
constexpr int kSmQF = 0;                             // Q fragments [16 k-steps][32 lanes] x 8 B
constexpr int kSmRowC = kSmQF + 16 * 32 * 8;         // c_row[8] floats
constexpr int kSmRed = kSmRowC + 128;                // reduction scratch (32 floats)
constexpr int kStages = 2;                           // copies in flight per warp: kStages - 1 blocks ahead
constexpr int kSmWarp = kSmRed + 128;                // per warp: kStages stage buffers
constexpr int kDecSmem = kSmWarp + kDecWarps * kStages * kStageBuf;
// combine area (aliases the stage buffers once every copy has landed)
constexpr int kCombFloats = 8 + 8 + 256 * 8;         // per warp: m[8], l[8], O^T[256][8]
static_assert(kDecWarps * kCombFloats * 4 <= kDecWarps * kStages * kStageBuf, "combine area fits the stage buffers");

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 8x8 b16 matrix held one row pair per thread (row lane/4, columns 2(lane%4),
// +1) -> its transpose in the same layout.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// Two int8 codes (bytes 0 and 1 of w) -> the f16 pair holding them exactly:
// byte b -> bits 0x64 | (b ^ 0x80) = 1024 + 128 + b as fp16, minus 1152.
__device__ __forceinline__ uint32_t codes2_to_f16x2(uint32_t w) {
  const uint32_t u = __byte_perm(w ^ 0x8080u, 0x6464u, 0x5140u);
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&u), __half2half2(__ushort_as_half(0x6480u)));
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Logical key block of the b-th visible block of a sequence.
__device__ __forceinline__ int dec_block(const DecSeq& d, int b) { return b < d.n_sink ? b : d.lo + (b - d.n_sink); }

__global__ void __launch_bounds__(kDecWarps * 32) decode_split_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int sp = blockIdx.x % p.max_splits;
  const int g = (blockIdx.x / p.max_splits) % p.HKV;
  const int s = blockIdx.x / (p.max_splits * p.HKV);
  const DecSeq ds = p.seqs[s];
  if (sp >= ds.n_splits) return;  // the whole CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int blk0 = sp * ds.per_split, blk1 = min(ds.n_vis, blk0 + ds.per_split);
  uint2* qf = reinterpret_cast<uint2*>(dsm + kSmQF);
  float* c_rows = reinterpret_cast<float*>(dsm + kSmRowC);

  // 1. The kv head's G query rows -> fp16 B fragments of Q^T, each row scaled
  // by the power of two that puts its absmax in [64, 128).  Thread: row r,
  // dims [16 c, 16 c + 16).  Rows >= G are zero.
  {
    const int r = threadIdx.x >> 4, c = threadIdx.x & 15;
    float v[16];
    float am = 0.f;
    if (r < p.G) {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)ds.q_row * p.HQ + (size_t)g * p.G + r) * kHeadDim +
                                                        c * 16);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 w = src[h];
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[8 * h + 2 * e] = __uint_as_float(ww[e] << 16);
          v[8 * h + 2 * e + 1] = __uint_as_float(ww[e] & 0xffff0000u);
        }
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) am = fmaxf(am, fabsf(v[e]));
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = 0.f;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const int k = am > 0.f ? min(127, 133 - (int)((__float_as_uint(am) >> 23) & 0xff)) : 0;
    const float mul = __uint_as_float((uint32_t)(127 + k) << 23);
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // dims 16c + 2i, +1: k-step c, column pair 2i
      const uint32_t pr = pack_f16x2(v[2 * i] * mul, v[2 * i + 1] * mul);
      uint2* slot = &qf[c * 32 + 4 * r + (i & 3)];
      if (i < 4) slot->x = pr;
      else slot->y = pr;
    }
    if (c == 0) c_rows[r] = r < p.G ? __uint_as_float((uint32_t)(127 - k) << 23) * p.sm_scale_log2 : 0.f;
  }
  __syncthreads();
  const float c_lo = c_rows[2 * tq], c_hi = c_rows[2 * tq + 1];

  // 2. This warp's blocks: blk0 + warp, + 4, ...  P' = p * v_scale * 2^-ev
  // with ev the exponent of the largest V scale the warp has met so far
  // (2^(ev-1) <= max < 2^ev, so P' <= 1); when a block raises it, O is
  // rescaled by the exact power of two, like the running max.
  const uint32_t stage0 = smem_u32(dsm + kSmWarp + warp * kStages * kStageBuf);
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  int ev = -100;
  float o[16][4];
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  // blocks of this warp: blk0 + warp + 4 i, i = 0 .. n_mine-1 (n_mine <= 32);
  // lane i holds block i's pool page, read once up front
  const int n_mine = blk1 > blk0 + warp ? (blk1 - blk0 - warp + kDecWarps - 1) / kDecWarps : 0;
  const int my_page = lane < n_mine ? p.block_table[(size_t)ds.bt_row * p.bt_stride +
                                                    dec_block(ds, blk0 + warp + kDecWarps * lane)]
                                    : -1;
  // copy block i's K and V codes (16 rows of 256 B each) and scales
  auto issue = [&](int i, uint32_t buf) -> bool {
    const int phys = __shfl_sync(0xffffffffu, my_page, i);
    if (phys < 0 || phys >= p.n_pool) return false;
    const size_t row0 = (size_t)phys * kPage * p.HKV + g;
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // 16 rows x 16 chunks of 16 B, K then V
      const int ch = lane + 32 * i, key = ch >> 4, cc = ch & 15;
      const size_t src = (row0 + (size_t)key * p.HKV) * kHeadDim + cc * 16;
      cp_async16(buf + key * kRowPitch + cc * 16, p.k_pool + src);
      cp_async16(buf + kStagePage + key * kRowPitch + cc * 16, p.v_pool + src);
    }
    const float* sc = lane < 16 ? p.k_scale : p.v_scale;
    cp_async4(buf + 2 * kStagePage + lane * 4, sc + row0 + (size_t)(lane & 15) * p.HKV);
    return true;
  };

  // block i goes to stage i % kStages
  uint32_t live_bits = 0;  // bit i: block i's page entry was in range
#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < n_mine && issue(i, stage0 + i * kStageBuf)) live_bits |= 1u << i;
    cp_async_commit();
  }
  for (int it = 0; it < n_mine; ++it) {
    const int b = blk0 + warp + kDecWarps * it;
    const uint32_t buf = stage0 + (it % kStages) * kStageBuf;
    const int ia = it + kStages - 1;  // the block whose copy goes out now
    if (ia < n_mine && issue(ia, stage0 + (ia % kStages) * kStageBuf)) live_bits |= 1u << ia;
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const bool live = (live_bits >> it) & 1u;
    if (!live) {
      if (lane == 0) atomicCAS(p.err, 0, DEV_ERR_BAD_PAGE);
    } else {
      const uint8_t* kb = dsm + (buf - smem_u32(dsm));
      const uint8_t* vb = kb + kStagePage;
      const float* scl = reinterpret_cast<const float*>(kb + 2 * kStagePage);
      // S^T = K Q^T: keys gq, gq+8 x rows 2tq, 2tq+1
      float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};  // even / odd k-steps
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const int d0 = 16 * kk + 2 * tq;
        uint32_t a[4];
        a[0] = codes2_to_f16x2(*reinterpret_cast<const uint16_t*>(kb + gq * kRowPitch + d0));
        a[1] = codes2_to_f16x2(*reinterpret_cast<const uint16_t*>(kb + (gq + 8) * kRowPitch + d0));
        a[2] = codes2_to_f16x2(*reinterpret_cast<const uint16_t*>(kb + gq * kRowPitch + d0 + 8));
        a[3] = codes2_to_f16x2(*reinterpret_cast<const uint16_t*>(kb + (gq + 8) * kRowPitch + d0 + 8));
        const uint2 bq = qf[kk * 32 + lane];
        if (kk & 1) mma16816(sacc2, a, bq.x, bq.y);
        else mma16816(sacc, a, bq.x, bq.y);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[e] += sacc2[e];
      // scores in log2 units; keys past the query position masked
      const int lb = dec_block(ds, b);
      const bool v0 = lb * kPage + gq <= ds.t, v1 = lb * kPage + gq + 8 <= ds.t;
      const float ks0 = scl[gq], ks1 = scl[gq + 8];
      const float y0 = v0 ? sacc[0] * ks0 * c_lo : -INFINITY, y1 = v0 ? sacc[1] * ks0 * c_hi : -INFINITY;
      const float y2 = v1 ? sacc[2] * ks1 * c_lo : -INFINITY, y3 = v1 ? sacc[3] * ks1 * c_hi : -INFINITY;
      float bm_lo = fmaxf(y0, y2), bm_hi = fmaxf(y1, y3);
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        bm_lo = fmaxf(bm_lo, __shfl_xor_sync(0xffffffffu, bm_lo, x));
        bm_hi = fmaxf(bm_hi, __shfl_xor_sync(0xffffffffu, bm_hi, x));
      }
      const float mn_lo = fmaxf(m_lo, bm_lo), mn_hi = fmaxf(m_hi, bm_hi);  // finite: key 0 of a block is visible
      // the block's largest V scale (scale slots 16..31 hold them)
      float bv = (lane >= 16 && lb * kPage + (lane - 16) <= ds.t) ? scl[lane] : 0.f;
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, x));
      const int evb = bv > 0.f ? max(-100, min(100, (int)((__float_as_uint(bv) >> 23) & 0xff) - 126)) : -100;
      // 2^(ev - evb) when the block raises ev; past 2^-126 the older terms are below fp32 resolution
      const int dev = evb - ev;
      const float vfix = dev <= 0 ? 1.f : (dev > 126 ? 0.f : __uint_as_float((uint32_t)(127 - dev) << 23));
      ev = max(ev, evb);
      const float vnorm = __uint_as_float((uint32_t)(127 - ev) << 23);
      const float al_lo = ex2f(m_lo - mn_lo), al_hi = ex2f(m_hi - mn_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      const float p0 = ex2f(y0 - mn_lo), p1 = ex2f(y1 - mn_hi), p2 = ex2f(y2 - mn_lo), p3 = ex2f(y3 - mn_hi);
      l_lo = l_lo * al_lo + (p0 + p2);
      l_hi = l_hi * al_hi + (p1 + p3);
      if (__any_sync(0xffffffffu, al_lo != 1.f || al_hi != 1.f || vfix != 1.f)) {
        const float f_lo = al_lo * vfix, f_hi = al_hi * vfix;
#pragma unroll
        for (int mt = 0; mt < 16; ++mt) {
          o[mt][0] *= f_lo;
          o[mt][1] *= f_hi;
          o[mt][2] *= f_lo;
          o[mt][3] *= f_hi;
        }
      }
      // P' = p * v_scale * 2^-ev (masked keys: 0, whatever their scale slot
      // holds), as the B fragments of P^T
      const float vs0 = v0 ? scl[16 + gq] * vnorm : 0.f, vs1 = v1 ? scl[16 + gq + 8] * vnorm : 0.f;
      const uint32_t pb0 = transpose8x8(pack_f16x2(v0 ? p0 * vs0 : 0.f, v0 ? p1 * vs0 : 0.f));
      const uint32_t pb1 = transpose8x8(pack_f16x2(v1 ? p2 * vs1 : 0.f, v1 ? p3 * vs1 : 0.f));
      // O^T += V^T P^T: dims 16 mt + gq (+8) x rows 2tq, 2tq+1
#pragma unroll
      for (int mt = 0; mt < 16; ++mt) {
        const int d = 16 * mt + gq;
        const uint8_t* r0 = vb + (2 * tq) * kRowPitch + d;
        const uint8_t* r8 = r0 + 8 * kRowPitch;
        uint32_t a[4];
        a[0] = codes2_to_f16x2((uint32_t)r0[0] | ((uint32_t)r0[kRowPitch] << 8));
        a[1] = codes2_to_f16x2((uint32_t)r0[8] | ((uint32_t)r0[kRowPitch + 8] << 8));
        a[2] = codes2_to_f16x2((uint32_t)r8[0] | ((uint32_t)r8[kRowPitch] << 8));
        a[3] = codes2_to_f16x2((uint32_t)r8[8] | ((uint32_t)r8[kRowPitch + 8] << 8));
        mma16816(o[mt], a, pb0, pb1);
      }
    }
    __syncwarp();  // every lane is done with this buffer before it is refilled
  }
  cp_async_wait<0>();
  // row sums over the warp's lanes that share tq
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, x);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, x);
  }
  __syncthreads();  // every warp's copies have landed: the stage area becomes the combine area

  // 3. Combine the four warps in shared memory into the split's partial.
  float* comb = reinterpret_cast<float*>(dsm + kSmWarp);
  float* mine = comb + warp * kCombFloats;
  if (gq == 0) {
    mine[2 * tq] = m_lo;
    mine[2 * tq + 1] = m_hi;
    mine[8 + 2 * tq] = l_lo;
    mine[8 + 2 * tq + 1] = l_hi;
  }
  const float vden = __uint_as_float((uint32_t)(127 + max(ev, -126)) << 23);  // O back to true V units: x 2^ev
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) {
    const int d = 16 * mt + gq;
    *reinterpret_cast<float2*>(mine + 16 + d * 8 + 2 * tq) = make_float2(o[mt][0] * vden, o[mt][1] * vden);
    *reinterpret_cast<float2*>(mine + 16 + (d + 8) * 8 + 2 * tq) = make_float2(o[mt][2] * vden, o[mt][3] * vden);
  }
  __syncthreads();
  for (int r = 0; r < p.G; ++r) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, comb[w * kCombFloats + r]);
    float wt[kDecWarps];
    float ls = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float mw = comb[w * kCombFloats + r];
      wt[w] = mw == -INFINITY ? 0.f : ex2f(mw - mx);
      ls += wt[w] * comb[w * kCombFloats + 8 + r];
    }
    float* part = p.part + (((size_t)s * p.HQ + (size_t)g * p.G + r) * p.max_splits + sp) * kDecPartStride;
    if (threadIdx.x == 0) {
      part[0] = mx;
      part[1] = ls;
    }
    for (int d = threadIdx.x; d < kHeadDim; d += kDecWarps * 32) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) acc += wt[w] * comb[w * kCombFloats + 16 + d * 8 + r];
      part[4 + d] = acc;
    }
  }
}

__global__ void __launch_bounds__(kHeadDim) decode_combine_kernel(const DecodeParams p) {
  const int s = blockIdx.x / p.HQ, h = blockIdx.x % p.HQ;
  const DecSeq ds = p.seqs[s];
  const float* part = p.part + ((size_t)s * p.HQ + h) * p.max_splits * kDecPartStride;
  float mx = -INFINITY;
  for (int i = 0; i < ds.n_splits; ++i) mx = fmaxf(mx, part[i * kDecPartStride]);
  float l = 0.f, acc = 0.f;
  const int d = threadIdx.x;
  for (int i = 0; i < ds.n_splits; ++i) {
    const float w = ex2f(part[i * kDecPartStride] - mx);
    l += w * part[i * kDecPartStride + 1];
    acc += w * part[i * kDecPartStride + 4 + d];
  }
  p.out[((size_t)ds.q_row * p.HQ + h) * kHeadDim + d] = __float2bfloat16_rn(l > 0.f ? acc / l : 0.f);
}

}  // namespace

int decode_ctas_per_sm() {
  static int n = 0;
  if (n <= 0) {
    if (cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel, kDecWarps * 32, kDecSmem) != cudaSuccess)
      n = 0;
    if (n <= 0) {
      (void)cudaGetLastError();
      n = 1;
    }
  }
  return n;
}

cudaError_t launch_decode(const DecodeParams& p, int n_seq, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
  if (e != cudaSuccess) return e;
  decode_split_kernel<<<n_seq * p.HKV * p.max_splits, kDecWarps * 32, kDecSmem, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  decode_combine_kernel<<<n_seq * p.HQ, kHeadDim, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
