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
// core.  So the int8 pool is read directly (no widening pass) and the small
// products run on warp-level MMAs (mma.sync m16n8k16, fp16 containers, fp32
// accumulate) in the transposed orientation, S^T = K Q^T and O^T = V^T P^T,
// so that keys and head dims fill M = 16 and the G query rows fill N = 8 with
// no padding.  In both the thread holds rows 2t, 2t+1 (t = lane % 4): the
// online-softmax state stays in registers.  Codes become exact fp16 pairs
// with byte permutes and one subtraction; the query enters as fp16 through a
// per-row power-of-two scale (lossless for bf16 input); P' = p * v_scale is
// normalised by the largest V scale the warp has met so far (a running power
// of two, rescaled like the running max) so that it stays in fp16's normal
// range.
//
// Data movement: each warp owns a ring of kDecStages block slots in shared
// memory; one lane fills them with TMA copies (a kv head's 16 token rows of a
// K page and of a V page, each as two 128-byte-swizzled halves), completing
// on the slot's mbarrier, so a warp has kDecStages blocks (kDecStages x 8 KB)
// in flight while it computes.  The page's 16 K and 16 V scales of the head
// come with them by 4-byte asynchronous copies, one per lane, into a 128-byte
// scale slot, tracked by the same mbarrier (cheaper than two more small bulk
// copies per block).
// Operand layout: the head dims of a block are permuted (the sum over dims in
// S^T is the same in any order; Q takes the same permutation, O^T is put back
// in order when written), so that every thread reads its K and V operands as
// 16-byte words of the swizzled rows instead of gathering bytes.
//
// Work split: the launch's (sequence, kv head) pairs laid end to end give one
// list of visible blocks; each CTA takes a run of it: runs of equal cost
// (blocks, plus a fixed charge for every pair a run crosses into) listed by
// the host in the launch parameters when one wave holds them, else equal runs
// over whole waves.  A CTA's run covers one or more segments (the part of a
// run that falls in one pair).  Per segment its 4 warps take the blocks in
// turn, then combine in shared memory in a fixed order (a call's result does
// not depend on scheduling): a segment that is a whole pair writes bf16 out
// directly; otherwise it writes a partial (row max, row sum, unnormalised O
// per q head) and adds its block count to the pair's ticket, and the CTA that
// completes the count merges the pair's partials and writes bf16 out.  The
// next segment's query rows are bulk-copied while the current one runs.
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
constexpr int kDecStages = 3;                        // block slots (copies in flight) per warp
constexpr int kHalfBytes = kPage * 128;              // 16 rows x 128 dims (one TMA box)
constexpr int kBlockBytes = 4 * kHalfBytes;          // K halves 0, 1, then V halves 0, 1
constexpr int kSlotsBytes = kDecWarps * kDecStages * kBlockBytes;
// Shared memory from a 1024-byte aligned base: the block slots, the Q
// fragments [16 k-steps][32 lanes] x 8 B (between segments: the combine
// area, 128 dims x 8 rows of fp32), small per-row values, the slots' barriers
// and the query rows' barrier, the slots' scales (lane l < 16: K scale of key
// l; 16 + l: V scale), and the raw bf16 query rows of the next segment
// (copied while the current one runs).
constexpr int kSmQf = kSlotsBytes;
constexpr int kSmMisc = kSmQf + 16 * 32 * 8;
constexpr int kSmBars = kSmMisc + 512;
constexpr int kSmQBar = kSmBars + kDecWarps * kDecStages * 8;
constexpr int kSmScales = kSmQBar + 16;
constexpr int kSmQRaw = kSmScales + kDecWarps * kDecStages * 128;
constexpr int kDecSmem = kSmQRaw + 8 * kHeadDim * 2 + 1024;
// Arrivals per slot phase: the copying lane's (with the byte count), then
// each lane's once its scale copy has landed.
constexpr int kSlotArrivals = 1 + 32;
// misc floats: row factors of Q [0, 8), per-warp row max / row sum [8, 72),
// the segment's row max / row sum [72, 88), the "last segment" flag at 88
constexpr int kMiscRowc = 0, kMiscWarp = 8, kMiscSeg = 72, kMiscFlag = 88;
constexpr uint64_t kDecDrainNs = 200000000ull;

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
// Codes held as (b ^ 0x80) in the low bytes of fp16 0x64__ are 1152 + b: the
// pair minus 1152 is the pair of codes, exactly.
__device__ __forceinline__ uint32_t f16x2_minus_1152(uint32_t u) {
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&u), __half2half2(__ushort_as_half(0x6480u)));
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Bytes 0, 1 (lo) or 2, 3 (hi) of a word of flipped codes (x = w ^ 0x80808080)
// as the fp16 pair 1152 + code (before the subtraction).
__device__ __forceinline__ uint32_t expand_lo(uint32_t x) { return __byte_perm(x, 0x64646464u, 0x5140); }
__device__ __forceinline__ uint32_t expand_hi(uint32_t x) { return __byte_perm(x, 0x64646464u, 0x7362); }
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
// 16-byte chunk c (0..7) of row r of a 128-byte-swizzled box: chunks are
// permuted by the row index mod 8, as the TMA copy writes them.
__device__ __forceinline__ uint32_t swz128(uint32_t half_base, int r, int c) {
  return half_base + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// A sequence's decode geometry (from the launch's table entry).
struct DecSeq {
  int q_row;   // row of the query token in q / out
  int t;       // its position in the context (n_ctx - 1)
  int vstart;  // visible blocks of the launch's earlier sequences (per kv head)
  int n_sink;  // sink blocks listed ahead of the window run
  int lo;      // first block of the window run (0 with the window off)
  int n_vis;   // visible blocks
};
__device__ __forceinline__ DecSeq dec_seq(const DecodeParams& p, const DecodeSeqs& tab, int s) {
  const int4 e = tab.seq[s];
  DecSeq d;
  d.q_row = e.x;
  d.t = e.y - 1;
  d.vstart = e.z;
  const int last = d.t / kPage;
  d.lo = p.W > 0 ? max(0, last + 1 - p.W) : 0;
  d.n_sink = p.W > 0 ? min(max(p.S, 0), d.lo) : 0;
  d.n_vis = d.n_sink + (last - d.lo + 1);
  return d;
}
// Logical key block of the b-th visible block of a sequence.
__device__ __forceinline__ int dec_block(const DecSeq& d, int b) { return b < d.n_sink ? b : d.lo + (b - d.n_sink); }

// Position of the pairs in the launch's block list: pair (s, g) starts at
// HKV vstart(s) + g n_vis(s).
struct PairPos {
  int s, g, start;
  DecSeq d;
};
// The pair that holds block x (0 <= x < total): the last sequence whose first
// block is at or before x (binary search over the table), then the kv head.
__device__ __forceinline__ PairPos dec_locate(const DecodeParams& p, const DecodeSeqs& tab, int x) {
  int lo = 0, hi = p.n_seq - 1;
  if (p.runs_listed) lo = hi = tab.cta_seq[blockIdx.x];  // x is this CTA's first block: the host found its sequence
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.HKV * tab.seq[mid].z <= x) lo = mid;
    else hi = mid - 1;
  }
  PairPos r;
  r.s = lo;
  r.d = dec_seq(p, tab, lo);
  r.g = (x - p.HKV * r.d.vstart) / r.d.n_vis;
  r.start = p.HKV * r.d.vstart + r.g * r.d.n_vis;
  return r;
}
__device__ __forceinline__ void dec_next_pair(const DecodeParams& p, const DecodeSeqs& tab, PairPos& r) {
  r.start += r.d.n_vis;
  if (++r.g == p.HKV) {
    r.g = 0;
    ++r.s;
    r.d = dec_seq(p, tab, r.s);
  }
}

// The kv head's G query rows (raw bf16 in shared memory) -> fp16 B fragments of Q^T, each row scaled by
// the power of two that puts its absmax in [64, 128).  Thread: row r, dims
// [16 c, 16 c + 16).  Rows >= G are zero.  Dims are permuted as the K operand
// is: k-step 4 j + m, lane (row, t) holds dims 64 j + 16 t + 4 m + {0, 1} and
// + {2, 3}.  Row factors (2^-k * sm_scale * log2 e) go to c_rows.
__device__ __forceinline__ void dec_load_q(const DecodeParams& p, const uint8_t* raw, uint2* qf, float* c_rows) {
  const int r = threadIdx.x >> 4, c = threadIdx.x & 15;
  float v[16];
  float am = 0.f;
  if (r < p.G) {
    const uint4* src = reinterpret_cast<const uint4*>(raw + r * kHeadDim * 2 + c * 32);
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
  for (int m = 0; m < 4; ++m)  // dims 16 c + 4 m + {0..3}: k-step 4 (c / 4) + m, lane (r, c % 4)
    qf[(4 * (c >> 2) + m) * 32 + 4 * r + (c & 3)] =
        make_uint2(pack_f16x2(v[4 * m] * mul, v[4 * m + 1] * mul), pack_f16x2(v[4 * m + 2] * mul, v[4 * m + 3] * mul));
  if (c == 0) c_rows[r] = r < p.G ? __uint_as_float((uint32_t)(127 - k) << 23) * p.sm_scale_log2 : 0.f;
}

__global__ void __launch_bounds__(kDecWarps * 32) decode_kernel(const __grid_constant__ DecodeParams p,
                                                                const __grid_constant__ DecodeSeqs tab,
                                                                const __grid_constant__ CUtensorMap km,
                                                                const __grid_constant__ CUtensorMap vm) {
  extern __shared__ uint8_t draw[];
  uint8_t* dsm = draw + ((1024u - (smem_u32(draw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(dsm);
  const int HKV = p.HKV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  uint2* qf = reinterpret_cast<uint2*>(dsm + kSmQf);
  float* comb = reinterpret_cast<float*>(dsm + kSmQf);  // between segments
  float* misc = reinterpret_cast<float*>(dsm + kSmMisc);
  const uint32_t bars = sbase + kSmBars;
  const WaitCtl wc{p.err, p.wait_ns};
  const uint32_t qbar = sbase + kSmQBar;
  if (threadIdx.x == 0) {
    mbar_init(qbar, 1);
    for (int i = 0; i < kDecWarps * kDecStages; ++i) mbar_init(bars + 8 * i, kSlotArrivals);
    fence_mbar_init();
    tma_prefetch_map(&km);
    tma_prefetch_map(&vm);
  }
  // this CTA's run of the launch's block list
  int x0, x1;
  if (p.runs_listed) {
    x0 = tab.cta_x0[blockIdx.x];
    x1 = blockIdx.x + 1 < gridDim.x ? tab.cta_x0[blockIdx.x + 1] : p.total;
  } else {
    x0 = (int)blockIdx.x * p.per_cta;
    x1 = min(p.total, x0 + p.per_cta);
  }
  PairPos pp = dec_locate(p, tab, x0);

  // 1. This warp's blocks: x0 + warp + 4 i, i < n_mine (<= 32).  Lane i looks
  // up block i's pool page and kv head once, walking the pairs from the
  // run's first.  Block i goes to slot i % kDecStages, whose barrier
  // completes once its copies landed.
  const int n_mine = x1 > x0 + warp ? (x1 - x0 - warp + kDecWarps - 1) / kDecWarps : 0;
  int my_page = -1, my_g = 0;
  if (lane < n_mine) {
    const int x = x0 + warp + kDecWarps * lane;
    PairPos q = pp;
    while (x >= q.start + q.d.n_vis) dec_next_pair(p, tab, q);
    my_g = q.g;
    my_page = p.block_table[(size_t)(p.bt_row0 + q.s) * p.bt_stride + dec_block(q.d, x - q.start)];
  }
  const uint32_t slot0 = sbase + (uint32_t)(warp * kDecStages * kBlockBytes);
  const uint32_t bar0 = bars + (uint32_t)(warp * kDecStages * 8);
  const uint32_t tx_bytes = (uint32_t)kBlockBytes;
  __syncthreads();  // the slots' barriers exist before any copy completes on them

  const uint32_t scl0 = sbase + (uint32_t)(kSmScales + warp * kDecStages * 128);
  // copy block i (a warp-wide call: page and kv head come from lane i); a
  // page entry outside the pool copies nothing and completes the slot's phase
  // at once.  Lane l < 16 copies the K scale of key l, lane 16 + l the V scale.
  auto issue = [&](int i) {
    const int phys = __shfl_sync(0xffffffffu, my_page, i);
    const int gi = __shfl_sync(0xffffffffu, my_g, i);
    const int st = i % kDecStages;
    const uint32_t bar = bar0 + 8 * st;
    if (phys < 0 || phys >= p.n_pool) {  // every lane arrives without a scale, lane 0 also for the copies
      mbar_arrive(bar);
      if (lane == 0) mbar_arrive(bar);
      return;
    }
    if (lane == 0) {
      const uint32_t dst = slot0 + (uint32_t)(st * kBlockBytes);
      mbar_expect_tx(bar, tx_bytes);
      tma_load_3d(dst, &km, bar, 0, gi, phys * kPage);
      tma_load_3d(dst + kHalfBytes, &km, bar, 128, gi, phys * kPage);
      tma_load_3d(dst + 2 * kHalfBytes, &vm, bar, 0, gi, phys * kPage);
      tma_load_3d(dst + 3 * kHalfBytes, &vm, bar, 128, gi, phys * kPage);
    }
    const float* src = (lane < 16 ? p.k_scale : p.v_scale) + ((size_t)phys * kPage + (lane & 15)) * HKV + gi;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(scl0 + (uint32_t)(st * 128 + lane * 4)), "l"(src)
                 : "memory");
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
  };
  // the first copies go out before the query setup, which they overlap
  int issued = min(kDecStages, n_mine);
  for (int i = 0; i < issued; ++i) issue(i);
  // a pair's G query rows (contiguous) into the raw area (thread 0)
  auto issue_q = [&](const PairPos& q) {
    const uint32_t bytes = (uint32_t)(p.G * kHeadDim * 2);
    mbar_expect_tx(qbar, bytes);
    bulk_load(sbase + kSmQRaw, p.q + ((size_t)q.d.q_row * p.HQ + (size_t)q.g * p.G) * kHeadDim, bytes, qbar);
  };
  bool q_pending = false;  // thread 0: a query copy not yet waited for
  bool q_broken = false;   // thread 0: a wait for one gave up
  if (threadIdx.x == 0) {
    issue_q(pp);
    q_pending = true;
  }
  uint32_t q_phase = 0;

  int it = 0;         // this warp's next block
  int waited = 0;     // blocks whose slot phase this warp has waited for
  bool ok = true;     // false once a wait gave up: the warp computes nothing more
  for (int x = x0; x < x1;) {  // segments
    const int seg_end = min(x1, pp.start + pp.d.n_vis);
    const DecSeq ds = pp.d;
    const int g = pp.g;
    // this segment's query rows (copied during the previous segment)
    const bool q_ok = mbar_wait(qbar, q_phase & 1u, wc, 61);
    ++q_phase;
    if (threadIdx.x == 0) {
      if (q_ok) q_pending = false;
      else q_broken = true;  // a copy may still be on its way: issue no other (one in flight at most)
    }
    if (!__all_sync(0xffffffffu, q_ok)) ok = false;
    dec_load_q(p, dsm + kSmQRaw, qf, misc + kMiscRowc);
    __syncthreads();  // the raw rows are read: the next segment's may come in
    if (threadIdx.x == 0 && seg_end < x1 && !q_broken) {
      PairPos nx = pp;
      dec_next_pair(p, tab, nx);
      issue_q(nx);
      q_pending = true;
    }
    const float c_lo = misc[kMiscRowc + 2 * tq], c_hi = misc[kMiscRowc + 2 * tq + 1];

    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    // P' = p * v_scale * 2^-ev with ev the exponent of the largest V scale the
    // warp has met so far in the segment (2^(ev-1) <= max < 2^ev, so P' <= 1);
    // when a block raises it, O is rescaled by the exact power of two, like
    // the running max.
    int ev = -100;
    float o[16][4];
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    // 2. The segment's blocks of this warp, in turn, as their copies land.
    for (; it < n_mine && x0 + warp + kDecWarps * it < seg_end; ++it) {
      const int st = it % kDecStages;
      if (ok && !__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * st, (uint32_t)(it / kDecStages) & 1u, wc, 60)))
        ok = false;
      if (!ok) continue;
      ++waited;
      const int b = x0 + warp + kDecWarps * it - pp.start;
      const int phys = __shfl_sync(0xffffffffu, my_page, it);
      if (phys < 0 || phys >= p.n_pool) {
        if (lane == 0) atomicCAS(p.err, 0, DEV_ERR_BAD_PAGE);
      } else {
        const uint32_t kb = slot0 + (uint32_t)(st * kBlockBytes), vb = kb + 2 * kHalfBytes;
        // S^T = K Q^T: keys gq, gq+8 x rows 2tq, 2tq+1.  Dims group j (64 dims,
        // 4 k-steps): this thread's 16 bytes of rows gq and gq+8, dims
        // 64 j + 16 tq + [0, 16); k-step 4 j + m takes word m (dims + 4m .. + 3).
        float sacc[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m) sacc[m][0] = sacc[m][1] = sacc[m][2] = sacc[m][3] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t hb = kb + (uint32_t)((j >> 1) * kHalfBytes);
          const int c = 4 * (j & 1) + tq;
          const uint4 r0 = lds128(swz128(hb, gq, c)), r1 = lds128(swz128(hb, gq + 8, c));
          const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t x0w = w0[m] ^ 0x80808080u, x1w = w1[m] ^ 0x80808080u;
            uint32_t a[4];
            a[0] = f16x2_minus_1152(expand_lo(x0w));
            a[1] = f16x2_minus_1152(expand_lo(x1w));
            a[2] = f16x2_minus_1152(expand_hi(x0w));
            a[3] = f16x2_minus_1152(expand_hi(x1w));
            const uint2 bq = qf[(4 * j + m) * 32 + lane];
            mma16816(sacc[m], a, bq.x, bq.y);  // four independent chains
          }
        }
        float sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = (sacc[0][e] + sacc[1][e]) + (sacc[2][e] + sacc[3][e]);
        // scores in log2 units; keys past the query position masked
        const int lb = dec_block(ds, b);
        const bool v0 = lb * kPage + gq <= ds.t, v1 = lb * kPage + gq + 8 <= ds.t;
        const float* scl = reinterpret_cast<const float*>(dsm + kSmScales) + (warp * kDecStages + st) * 32;
        const float ks0 = scl[gq], ks1 = scl[gq + 8], vsc0 = scl[16 + gq], vsc1 = scl[24 + gq];
        const float y0 = v0 ? sc[0] * ks0 * c_lo : -INFINITY, y1 = v0 ? sc[1] * ks0 * c_hi : -INFINITY;
        const float y2 = v1 ? sc[2] * ks1 * c_lo : -INFINITY, y3 = v1 ? sc[3] * ks1 * c_hi : -INFINITY;
        float bm_lo = fmaxf(y0, y2), bm_hi = fmaxf(y1, y3);
        // the block's largest V scale (lanes 16..31: the V scales of keys 0..15)
        float bv = (lane >= 16 && lb * kPage + (lane - 16) <= ds.t) ? scl[lane] : 0.f;
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
          bm_lo = fmaxf(bm_lo, __shfl_xor_sync(0xffffffffu, bm_lo, sh));
          bm_hi = fmaxf(bm_hi, __shfl_xor_sync(0xffffffffu, bm_hi, sh));
          bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, sh));
        }
        bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, 2));
        bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, 1));
        const float mn_lo = fmaxf(m_lo, bm_lo), mn_hi = fmaxf(m_hi, bm_hi);  // finite: key 0 of a block is visible
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
        const float vs0 = v0 ? vsc0 * vnorm : 0.f, vs1 = v1 ? vsc1 * vnorm : 0.f;
        const uint32_t pb0 = transpose8x8(pack_f16x2(v0 ? p0 * vs0 : 0.f, v0 ? p1 * vs0 : 0.f));
        const uint32_t pb1 = transpose8x8(pack_f16x2(v1 ? p2 * vs1 : 0.f, v1 ? p3 * vs1 : 0.f));
        // O^T += V^T P^T.  Dims are permuted: row gq of m-tile mt is dim
        // 32 gq + 2 mt, row gq + 8 is dim 32 gq + 2 mt + 1, so this thread's A
        // operands come from dims [32 gq, 32 gq + 32) of keys 2tq, 2tq+1, 2tq+8,
        // 2tq+9: words i (dims 32 gq + 4 i .. + 3) feed m-tiles 2i and 2i+1.
        // Bytes of a key pair are interleaved first ([k.d, k'.d, k.d+1, k'.d+1]),
        // then each half widens to the fp16 pair (key, key') of one dim.
        const uint32_t vh = vb + (uint32_t)((gq >> 2) * kHalfBytes);
        const int key[4] = {2 * tq, 2 * tq + 1, 2 * tq + 8, 2 * tq + 9};
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // dims 32 gq + 16 h .. + 15: words i = 4 h .. 4 h + 3
          uint32_t w[4][4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 r = lds128(swz128(vh, key[k], 2 * (gq & 3) + h));
            w[k][0] = r.x, w[k][1] = r.y, w[k][2] = r.z, w[k][3] = r.w;
          }
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) {
            const int i = 4 * h + ii;
            const uint32_t lo01 = __byte_perm(w[0][ii], w[1][ii], 0x5140) ^ 0x80808080u;  // dims + 0, + 1
            const uint32_t hi01 = __byte_perm(w[0][ii], w[1][ii], 0x7362) ^ 0x80808080u;  // dims + 2, + 3
            const uint32_t lo89 = __byte_perm(w[2][ii], w[3][ii], 0x5140) ^ 0x80808080u;
            const uint32_t hi89 = __byte_perm(w[2][ii], w[3][ii], 0x7362) ^ 0x80808080u;
            uint32_t a[4];
            // m-tile 2i: dims + 0 (row gq) and + 1 (row gq + 8); keys (2tq, 2tq+1) and (2tq+8, 2tq+9)
            a[0] = f16x2_minus_1152(expand_lo(lo01));
            a[1] = f16x2_minus_1152(expand_hi(lo01));
            a[2] = f16x2_minus_1152(expand_lo(lo89));
            a[3] = f16x2_minus_1152(expand_hi(lo89));
            mma16816(o[2 * i], a, pb0, pb1);
            // m-tile 2i+1: dims + 2 and + 3
            a[0] = f16x2_minus_1152(expand_lo(hi01));
            a[1] = f16x2_minus_1152(expand_hi(hi01));
            a[2] = f16x2_minus_1152(expand_lo(hi89));
            a[3] = f16x2_minus_1152(expand_hi(hi89));
            mma16816(o[2 * i + 1], a, pb0, pb1);
          }
        }
      }
      __syncwarp();  // every lane is done with this slot before it is refilled
      if (it + kDecStages < n_mine) {
        issue(it + kDecStages);
        ++issued;
      }
    }
    // row sums over the warp's lanes that share tq
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      l_lo += __shfl_xor_sync(0xffffffffu, l_lo, sh);
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, sh);
    }
    float* wml = misc + kMiscWarp;
    if (gq == 0) {
      wml[warp * 16 + 2 * tq] = m_lo;
      wml[warp * 16 + 2 * tq + 1] = m_hi;
      wml[warp * 16 + 8 + 2 * tq] = l_lo;
      wml[warp * 16 + 8 + 2 * tq + 1] = l_hi;
    }
    __syncthreads();  // every warp is done with the segment: its Q fragments area becomes the combine area

    // 3. Combine the warps: this thread's rows 2tq, 2tq+1; the segment's row
    // max and sum; each warp's factor (2^(m_w - max) and O back to true V
    // units, x 2^ev).  A warp without blocks here has m = -inf and O = 0.
    float f[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 2 * tq + e;
      float mx = -INFINITY, ls = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, wml[w * 16 + r]);
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = wml[w * 16 + r];
        ls += mw == -INFINITY ? 0.f : ex2f(mw - mx) * wml[w * 16 + 8 + r];
      }
      const float mine = e ? m_hi : m_lo;
      f[e] = mine == -INFINITY ? 0.f : ex2f(mine - mx) * __uint_as_float((uint32_t)(127 + max(ev, -126)) << 23);
      if (warp == 0 && gq == 0) {
        misc[kMiscSeg + r] = mx;
        misc[kMiscSeg + 8 + r] = ls;
      }
    }
    const int pair = pp.s * HKV + g;
    const bool whole = x == pp.start && seg_end == pp.start + ds.n_vis;
    // a later segment of the run starts its pair: the pair's first CTA
    const int slot = x != x0 ? 0 : (p.runs_listed ? (int)tab.cta_slot[blockIdx.x] : (int)blockIdx.x - pp.start / p.per_cta);
    float* part = p.part + ((size_t)pair * p.max_slots + slot) * p.G * kDecPartStride;
    __nv_bfloat16* out = p.out + ((size_t)ds.q_row * p.HQ + (size_t)g * p.G) * kHeadDim;
    // Two rounds of 128 dims through the combine area, word (2 jj + e) * 32 +
    // 4 gq + tq for row 2tq + e, dim 32 gq + 16 h + jj (jj = 2 (mt - 8 h) + {0, 1}):
    // warp 0 stores, then warps 1, 2, 3 add in turn (a fixed order: the same
    // inputs give the same bits); then thread (gq = t % 8, jj = t / 8) reads
    // its dim's 8 rows as two float4.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        if (warp == w) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float* oo = o[8 * h + q];
            float* cw = comb + (4 * q) * 32 + 4 * gq + tq;  // jj = 2q: words 2jj, 2jj+1; jj = 2q+1: 2jj+2, 2jj+3
            const float v0 = oo[0] * f[0], v1 = oo[1] * f[1], v2 = oo[2] * f[0], v3 = oo[3] * f[1];
            if (w == 0) {
              cw[0] = v0;
              cw[32] = v1;
              cw[64] = v2;
              cw[96] = v3;
            } else {
              cw[0] += v0;
              cw[32] += v1;
              cw[64] += v2;
              cw[96] += v3;
            }
          }
        }
        __syncthreads();
      }
      {
        const int rg = threadIdx.x & 7, jj = threadIdx.x >> 3;
        const int d = 32 * rg + 16 * h + jj;
        const float4 ev4 = *reinterpret_cast<const float4*>(comb + (2 * jj) * 32 + 4 * rg);      // rows 0, 2, 4, 6
        const float4 od4 = *reinterpret_cast<const float4*>(comb + (2 * jj + 1) * 32 + 4 * rg);  // rows 1, 3, 5, 7
        const float val[8] = {ev4.x, od4.x, ev4.y, od4.y, ev4.z, od4.z, ev4.w, od4.w};
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r >= p.G) break;
          if (whole) out[(size_t)r * kHeadDim + d] = __float2bfloat16_rn(val[r] / misc[kMiscSeg + 8 + r]);
          else part[(size_t)r * kDecPartStride + 4 + d] = val[r];
        }
        if (!whole && h == 0 && threadIdx.x < p.G) {
          part[(size_t)threadIdx.x * kDecPartStride] = misc[kMiscSeg + threadIdx.x];
          part[(size_t)threadIdx.x * kDecPartStride + 1] = misc[kMiscSeg + 8 + threadIdx.x];
        }
      }
      __syncthreads();
    }

    // 4. A partial: count its blocks in; the CTA that completes the pair
    // merges every partial of it.  Ordering: the CTA's partial writes come
    // before the barrier the loop above ended with, thread 0's fence makes
    // them visible at device scope before its ticket add (release), and its
    // fence after the add orders the merge's reads after it (acquire).
    if (!whole) {
      if (threadIdx.x == 0) {
        __threadfence();
        // blocks, and (from the pair's last CTA) the partial count
        const unsigned long long add = (unsigned long long)(seg_end - x) +
            (seg_end == pp.start + ds.n_vis ? (unsigned long long)(slot + 1) << 32 : 0ull);
        const unsigned long long now = atomicAdd(&p.tickets[pair], add) + add;
        const bool last = (uint32_t)now == (uint32_t)ds.n_vis;
        if (last) p.tickets[pair] = 0;  // every other CTA of the pair has counted in: reset for the next launch
        __threadfence();
        reinterpret_cast<int*>(misc)[kMiscFlag] = last ? (int)(now >> 32) : 0;
      }
      __syncthreads();
      const int n_sl = reinterpret_cast<const int*>(misc)[kMiscFlag];
      if (n_sl > 0) {
        // thread (row t / 16, dims 16 (t % 16) .. + 15): the pair's partials
        // four at a time (all their loads in flight together), merged online
        const int r = threadIdx.x >> 4, dc = (threadIdx.x & 15) * 16;
        if (r < p.G) {
          const size_t sstride = (size_t)p.G * kDecPartStride;
          const float* pr = p.part + (size_t)pair * p.max_slots * sstride + (size_t)r * kDecPartStride;
          float mx = -INFINITY, l = 0.f;
          float acc[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] = 0.f;
          for (int k0 = 0; k0 < n_sl; k0 += 4) {
            float mk[4], lk[4];
            float4 ok[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const bool have = k0 + u < n_sl;
              const float* ps = pr + (size_t)(have ? k0 + u : k0) * sstride;
              mk[u] = have ? __ldcg(ps) : -INFINITY;
              lk[u] = __ldcg(ps + 1);
#pragma unroll
              for (int e = 0; e < 4; ++e) ok[u][e] = __ldcg(reinterpret_cast<const float4*>(ps + 4 + dc) + e);
            }
            float mn = mx;
#pragma unroll
            for (int u = 0; u < 4; ++u) mn = fmaxf(mn, mk[u]);
            const float al = mx == -INFINITY ? 0.f : ex2f(mx - mn);
            l *= al;
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] *= al;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float w = mk[u] == -INFINITY ? 0.f : ex2f(mk[u] - mn);
              l += w * lk[u];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc[4 * e] += w * ok[u][e].x;
                acc[4 * e + 1] += w * ok[u][e].y;
                acc[4 * e + 2] += w * ok[u][e].z;
                acc[4 * e + 3] += w * ok[u][e].w;
              }
            }
            mx = mn;
          }
          const float il = l > 0.f ? 1.f / l : 0.f;
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * e] * il, acc[2 * e + 1] * il);
            pk[e] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(out + (size_t)r * kHeadDim + dc);
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
    x = seg_end;
    if (x < x1) dec_next_pair(p, tab, pp);
    __syncthreads();  // the combine area is free before the next segment's Q fragments
  }
  // every copy this warp issued lands before the CTA exits (after a wait gave
  // up some were never waited for; bounded)
  if (threadIdx.x == 0 && q_pending) (void)mbar_wait_drain(qbar, (q_phase - 1u) & 1u, kDecDrainNs);
  if (lane == 0)
    for (int i = waited; i < issued; ++i)
      (void)mbar_wait_drain(bar0 + 8 * (i % kDecStages), (uint32_t)(i / kDecStages) & 1u, kDecDrainNs);
  __syncwarp();
}

}  // namespace

int decode_ctas_per_sm(int HKV) {
  static int cached[9] = {0};
  if (HKV < 1 || HKV > 8) return 1;
  int& n = cached[HKV];
  if (n <= 0) {
    if (cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel, kDecWarps * 32, kDecSmem) != cudaSuccess)
      n = 0;
    if (n <= 0) {
      (void)cudaGetLastError();
      n = 1;
    }
  }
  return n;
}

cudaError_t launch_decode(const DecodeParams& p, const DecodeSeqs& seqs, const DecodeMaps& m, int n_cta,
                          cudaStream_t st) {
  const cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
  if (e != cudaSuccess) return e;
  decode_kernel<<<n_cta, kDecWarps * 32, kDecSmem, st>>>(p, seqs, m.k, m.v);
  return cudaGetLastError();
}

}  // namespace pa
