// Gather-side kernels of the windowed prefill attention over a paged int8 KV
// pool (sm_103a):
//
//   widen_kernel      page gather through the block table: int8 K/V pages ->
//                     contiguous integer-valued copies (K row-major in bf16, V
//                     transposed in fp16) plus per-token scales, visible blocks only.
//   debug kernels     exports of the gather and of the mask set for the tests,
//                     built on the same geometry helpers as the attention kernel.
//
// sm_103a has no integer tcgen05 MMA, so the int8 codes are widened once per
// call into 16-bit float containers (exact: |code| <= 127) that the attention
// kernel (pa_attention.cu) feeds to tcgen05.mma kind::f16: K in bf16, the type
// of Q, and V in fp16, the type of P'.
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

// One CTA per stored 16-token block.  Every load of the block (its K and V
// codes, HKV x 16-byte chunks each per thread, and its scales) is issued
// before the first store: the stores go to other arrays, but the compiler
// cannot tell, and a load behind each store would leave one load in flight
// per thread (the kernel is bound by load latency, not by bandwidth).
template <int HKV>
__global__ void __launch_bounds__(kWidenThreads) widen_kernel(const WidenParams p) {
  __shared__ __align__(16) int8_t vpage[kPage * HKV * kHeadDim];
  __shared__ unsigned int vmax_sh[HKV];  // the block's largest V scale per head (bit pattern)
  const int blk = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < HKV) vmax_sh[tid] = 0u;
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
  const size_t page_base = (size_t)(bad ? 0 : phys) * kPage * HKV * kHeadDim;

  // loads: chunk idx = tid + 256 i is bytes [16 idx, 16 idx + 16) of the
  // page, i.e. token idx / (16 HKV), head (idx / 16) % HKV, dims 16 (idx % 16) on
  int4 kr[HKV], vr[HKV];
#pragma unroll
  for (int i = 0; i < HKV; ++i) {
    const int idx = tid + kWidenThreads * i;
    kr[i] = vr[i] = make_int4(0, 0, 0, 0);
    if (idx / (HKV * 16) < n_valid) {
      kr[i] = __ldg(reinterpret_cast<const int4*>(p.k_pool + page_base) + idx);
      vr[i] = __ldg(reinterpret_cast<const int4*>(p.v_pool + page_base) + idx);
    }
  }
  float ksv = 0.f, vsv = 0.f;  // thread tid < 16 HKV: token tid / HKV, head tid % HKV
  if (tid < kPage * HKV && tid / HKV < n_valid) {
    const size_t slot = ((size_t)phys * kPage + tid / HKV) * HKV + tid % HKV;
    ksv = __ldg(p.k_scale + slot);
    vsv = __ldg(p.v_scale + slot);
  }

  // K: each chunk's 16 codes as bf16, at its row of the head's widened K
#pragma unroll
  for (int i = 0; i < HKV; ++i) {
    const int idx = tid + kWidenThreads * i;
    const int c = idx & 15, g = (idx >> 4) % HKV, tk = (idx >> 4) / HKV;
    const int8_t* cb = reinterpret_cast<const int8_t*>(&kr[i]);
    __align__(16) __nv_bfloat16 h[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) h[e] = __int2bfloat16_rn((int)cb[e]);
    int4* dst = reinterpret_cast<int4*>(p.kw + ((size_t)g * p.n_tok_cap + row0 + tk) * kHeadDim + c * 16);
    dst[0] = reinterpret_cast<const int4*>(h)[0];
    dst[1] = reinterpret_cast<const int4*>(h)[1];
  }
  // V: stage the page, then write each (head, dim) column of 16 tokens
#pragma unroll
  for (int i = 0; i < HKV; ++i) reinterpret_cast<int4*>(vpage)[tid + kWidenThreads * i] = vr[i];
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
  // scales (0 past the end of the context) and the running max of V scales:
  // reduced in the block first, then one global atomic per head, and only
  // when it raises the maximum (thousands of blocks update the same words)
  if (tid < kPage * HKV) {
    const int tk = tid / HKV, g = tid % HKV;
    p.ks[(size_t)g * p.n_tok_cap + row0 + tk] = ksv * p.k_mult;
    p.vs[(size_t)g * p.n_tok_cap + row0 + tk] = vsv;
    if (vsv > 0.f) atomicMax(&vmax_sh[g], __float_as_uint(vsv));
  }
  __syncthreads();
  if (tid < HKV) {
    const unsigned int m = vmax_sh[tid];
    unsigned int* gm = p.vsmax + s * HKV + tid;
    if (m > *reinterpret_cast<volatile unsigned int*>(gm)) atomicMax(gm, m);
  }
}

cudaError_t launch_widen(const WidenParams& p, cudaStream_t st) {
  switch (p.HKV) {
    case 1: widen_kernel<1><<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p); break;
    case 2: widen_kernel<2><<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p); break;
    case 3: widen_kernel<3><<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p); break;
    case 4: widen_kernel<4><<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p); break;
    case 5: widen_kernel<5><<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p); break;
    case 6: widen_kernel<6><<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p); break;
    case 7: widen_kernel<7><<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p); break;
    case 8: widen_kernel<8><<<p.n_stored_blocks, kWidenThreads, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;  // the handle accepts 1..8 kv heads
  }
  return cudaGetLastError();
}

// ======================================================================
// KV append: the step before the path.  Each new (token, kv head) row of K
// and of V is quantised symmetrically on its own (scale = absmax / 127, code
// = rint(x / scale) half to even, clamped to [-127, 127], all in fp32 with
// correctly rounded divisions; an all-zero row gets scale 0) and written into
// its pool slot: page bt_row[tok / 16], slot tok % 16.
// One warp per new token: its 2 x HKV rows (K and V of every kv head), 8
// values per lane per row, all rows' loads in flight before any reduction.
constexpr int kAppendWarps = 8;

// |x| of a lane's eight bf16 values, as the bit pattern of their largest
// magnitude (non-negative bf16 patterns order like their values).
__device__ __forceinline__ uint32_t absmax_bits8(const uint4 raw) {
  const uint32_t m = __vmaxu2(__vmaxu2(raw.x & 0x7fff7fffu, raw.y & 0x7fff7fffu),
                              __vmaxu2(raw.z & 0x7fff7fffu, raw.w & 0x7fff7fffu));
  return max(m & 0xffffu, m >> 16);
}

// Quantise a lane's eight bf16 values of a row whose absolute maximum over
// the warp is `am`: codes rint(x / scale) half to even, scale = absmax / 127.
__device__ __forceinline__ uint2 quantise_row8(const uint4 raw, float am, float& scale_out) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
  }
  // scale = RN(am / 127) without a division: Markstein's division by a
  // constant (q0 = RN(am r), r = RN(1/127); the remainder am - 127 q0 is exact
  // in one FMA; q1 = RN(q0 + rem r)).  Checked exhaustively: for every
  // positive finite bf16 magnitude the remainder is representable and q1 is
  // the correctly rounded quotient.
  constexpr float kInv127 = 1.0f / 127.0f;
  const float q0 = __fmul_rn(am, kInv127);
  const float scale = __fmaf_rn(__fmaf_rn(-q0, 127.f, am), kInv127, q0);
  // code = rint(x / scale) on the IEEE-rounded quotient.  x * rcp, with rcp
  // the hardware reciprocal (within 1 ulp), is within 3.1e-5 of that quotient
  // (|quotient| <= 127.5), so where it is farther than 1e-4 from a
  // half-integer both round the same way; near one the division itself
  // decides.  |code| <= 127 without a clamp: |x| <= absmax and scale =
  // RN(absmax / 127), so |x / scale| <= 127 (1 + 2^-23).  Adding 1.5 * 2^23
  // rounds a value of magnitude < 2^22 to an integer, ties to even, and the
  // sum's low byte is that integer's two's complement byte: the code.
  float rcp = 0.f;
  if (scale > 0.f) asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rcp) : "f"(scale));
  constexpr float kRound = 12582912.f;  // 1.5 * 2^23
  uint32_t f[8];
  float dmax = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 q = mul2(make_float2(x[2 * e], x[2 * e + 1]), make_float2(rcp, rcp));
    const float2 fr = add2(q, make_float2(kRound, kRound));
    const float2 r = add2(fr, make_float2(-kRound, -kRound));
    const float2 d = add2(q, make_float2(-r.x, -r.y));
    dmax = max3(dmax, fabsf(d.x), fabsf(d.y));
    f[2 * e] = __float_as_uint(fr.x);
    f[2 * e + 1] = __float_as_uint(fr.y);
  }
  // A quotient near a half-integer is rounded from the division (rare), and so
  // is every quotient of a row with a subnormal scale (absmax < 127 * 2^-126),
  // whose reciprocal the approximate instruction cannot give.
  if (dmax > 0.4999f || (scale > 0.f && scale < 1.17549435e-38f)) {
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = __float_as_uint(rintf(__fdiv_rn(x[e], scale)) + kRound);
  }
  // low bytes of the sums, four to a word
  const uint32_t lo = __byte_perm(__byte_perm(f[0], f[1], 0x0040), __byte_perm(f[2], f[3], 0x0040), 0x5410);
  const uint32_t hi = __byte_perm(__byte_perm(f[4], f[5], 0x0040), __byte_perm(f[6], f[7], 0x0040), 0x5410);
  scale_out = scale;
  return make_uint2(lo, hi);
}

// Six blocks per SM (40 registers): more warps to cover the loads; measured
// ~5 % faster than the five that 43 registers allow.
template <int HKV>
__global__ void __launch_bounds__(kAppendWarps * 32, 6) kv_append_kernel(const KvAppendParams p) {
  const int i = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);  // new token
  const int lane = threadIdx.x & 31;
  if (i >= p.n_new) return;
  const int tok = p.tok_start + i;
  // the rows' loads go out with the block-table read, not after it
  const int phys = p.bt_row[tok / kPage];
  const size_t row0 = (size_t)i * HKV;
  uint4 rk[HKV], rv[HKV];
#pragma unroll
  for (int g = 0; g < HKV; ++g) {
    rk[g] = reinterpret_cast<const uint4*>(p.k_new + (row0 + g) * kHeadDim)[lane];
    rv[g] = reinterpret_cast<const uint4*>(p.v_new + (row0 + g) * kHeadDim)[lane];
  }
  if (phys < 0 || phys >= p.n_pool) {  // never dereferenced
    if (lane == 0) atomicCAS(p.err, 0, DEV_ERR_BAD_PAGE);
    return;
  }
  const size_t slot0 = ((size_t)phys * kPage + tok % kPage) * HKV;
#pragma unroll
  for (int g = 0; g < HKV; ++g) {
      // the K and V rows' absolute maxima reduced over the warp together, as
      // the two 16-bit halves of one word (each is a bf16 magnitude)
      uint32_t m2 = absmax_bits8(rk[g]) | (absmax_bits8(rv[g]) << 16);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, o));
      float sk, sv;
      const uint2 ck = quantise_row8(rk[g], __uint_as_float(m2 << 16), sk);
      const uint2 cv = quantise_row8(rv[g], __uint_as_float(m2 & 0xffff0000u), sv);
      reinterpret_cast<uint2*>(p.k_pool + (slot0 + g) * kHeadDim)[lane] = ck;
      reinterpret_cast<uint2*>(p.v_pool + (slot0 + g) * kHeadDim)[lane] = cv;
      if (lane == 0) {
        p.k_scale[slot0 + g] = sk;
        p.v_scale[slot0 + g] = sv;
      }
    }
}

cudaError_t launch_kv_append(const KvAppendParams& p, cudaStream_t st) {
  if (p.n_new <= 0) return cudaSuccess;
  const int grid = (p.n_new + kAppendWarps - 1) / kAppendWarps;
  switch (p.HKV) {
    case 1: kv_append_kernel<1><<<grid, kAppendWarps * 32, 0, st>>>(p); break;
    case 2: kv_append_kernel<2><<<grid, kAppendWarps * 32, 0, st>>>(p); break;
    case 3: kv_append_kernel<3><<<grid, kAppendWarps * 32, 0, st>>>(p); break;
    case 4: kv_append_kernel<4><<<grid, kAppendWarps * 32, 0, st>>>(p); break;
    case 5: kv_append_kernel<5><<<grid, kAppendWarps * 32, 0, st>>>(p); break;
    case 6: kv_append_kernel<6><<<grid, kAppendWarps * 32, 0, st>>>(p); break;
    case 7: kv_append_kernel<7><<<grid, kAppendWarps * 32, 0, st>>>(p); break;
    case 8: kv_append_kernel<8><<<grid, kAppendWarps * 32, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;  // the handle accepts 1..8 kv heads
  }
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
          (int8_t)__bfloat162int_rn(p.kw[((size_t)g * p.n_tok_cap + row) * kHeadDim + d]);
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
__global__ void debug_maskset_kernel(const SeqGeom* seqs, const Unit* units, int UT, int G, int S, int W,
                                     int32_t* row_counts, int32_t* unit_blocks, int cap) {
  const Unit un = units[blockIdx.x];
  const SeqGeom sg = seqs[un.seq];
  const UnitGeom ug = unit_geom(un.t0, UT, sg, S, W);
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
    count += __popcll(visible_columns(tg, t_row, S, W, 0)) + __popcll(visible_columns(tg, t_row, S, W, 1));
  }
  if (r == 0)
    for (int k = nblk; k < cap; ++k) unit_blocks[(size_t)blockIdx.x * cap + k] = -1;
  row_counts[(size_t)blockIdx.x * kUnitRows + r] = count;
}

cudaError_t launch_debug_maskset(const SeqGeom* seqs, const Unit* units, int n_units, int UT, int G, int S, int W,
                                 int32_t* row_counts, int32_t* unit_blocks, int cap, cudaStream_t st) {
  debug_maskset_kernel<<<n_units, kUnitRows, 0, st>>>(seqs, units, UT, G, S, W, row_counts, unit_blocks, cap);
  return cudaGetLastError();
}

}  // namespace pa
