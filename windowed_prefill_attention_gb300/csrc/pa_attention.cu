// Attention kernel of the windowed prefill attention over a paged int8 KV pool
// (sm_103a): a persistent, warp-specialised tcgen05 pipeline.
//
// The method ("int8 tensor-core prefill attention", sections "Summary" and
// "Why the attention, and why tensor cores"): the query quantised per row in
// a fused prologue; QK^T on the tensor cores over K codes read from the paged
// pool; the per-row Q, per-token K and softmax scales applied to the integer-
// valued scores; the online-softmax recurrence; the per-token V scale folded
// into P before P is quantised per row; PV on the tensor cores; masked blocks
// never visited.  The int8 codes travel in 16-bit float containers
// (tcgen05.mma kind::f16), which hold them exactly: K in bf16 against the bf16
// query, V in fp16 against P' in fp16.
//
// Pairs of SMs (clusters of two CTAs, one per SM) each take the units the
// host handed them (longest first, each to the pair with the least work so
// far), or walk the list with stride = the number of pairs.  A unit is 256
// query rows of one kv head (pa_tiles.cuh), 128 in each CTA; one 256-row tcgen05 MMA
// (cta_group::2, issued by the even CTA) covers both, with the B operand (K
// keys for QK^T, V^T dims for PV) split between the two CTAs' shared memory,
// so each SM stores and reads only half of every K/V tile.  Key tiles are
// 128 keys; with N = 128 a QK^T instruction runs at the tensor core's full
// rate (at N = 64 it does not), which sets the memory plan, per CTA:
//   TMEM (512 columns)   O fp32 [0,256), S0 [256,384), S1 [384,512) for the
//                        CTA's 128 rows; P' (fp16 pairs) of softmax half h
//                        overwrites S columns [64h, 64h+32)
//   shared memory        Q (64 KB, bf16, TMA), K as 2 x 4 slots of 8 KB (tile
//                        parity x 64-dim region; this CTA's 64 keys), V^T as
//                        2 x 2 slots of 16 KB (tile parity x 64-key chunk;
//                        this CTA's 128 dims), the tiles' K/V scales in two
//                        1 KB slots
// K and V^T are double-buffered by tile parity, so the MMA issuer waits once
// per operand per tile.  Roles (both CTAs unless noted):
//   warp 0        TMA producer of K (one lane per slot); the odd CTA's copies
//                 complete on the even CTA's barrier
//   warp 1        TMEM allocator (for the pair); in the even CTA the single
//                 MMA-issuing thread; QK^T(j+1) is issued before PV(j), so the
//                 tensor core works on the next scores while the softmax
//                 handles the current ones
//   warp 2        TMA producer of V^T (one lane per slot), as warp 0
//   warp 3        producer of Q (TMA, one lane per region, after an L2
//                 prefetch) and of the scales
//   warps 4-11    softmax: two warps per TMEM lane quadrant, each owning 16
//                 whole rows (two rows per thread, 16-lane TMEM shapes)
//   warps 12-15   epilogue of each unit (and Q codes on the int8 grid)
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kSlices = 2;                              // softmax warps per TMEM lane quadrant (16 rows each)
constexpr int kSoftmaxWarps = 4 * kSlices;             // warps 4 .. 11
constexpr int kThreads = 32 * (4 + kSoftmaxWarps + 4);  // + producers/MMA (0-3) and epilogue (12-15)
constexpr int kRegionBytes = kRows * 128;                 // 16 KB: Q, 128 rows x 64 dims (bf16)
constexpr int kKSlotBytes = (kTileKeys / 2) * 128;        // 8 KB: this CTA's 64 keys x 64 dims (bf16)
constexpr int kVSlotBytes = (kHeadDim / 2) * kChunkKeys * 2;  // 16 KB: this CTA's 128 dims x 64 keys (fp16)
constexpr int kKSlots = 8;                                // [tile parity][64-dim region]
constexpr int kVSlots = 4;                                // [tile parity][64-key chunk]
// Shared memory, offsets from a 1024-byte aligned base (the same in both CTAs).
constexpr int kSmQ = 0;                                   // 4 regions of 128 rows x 128 B
constexpr int kSmK = kSmQ + 4 * kRegionBytes;             // K slots
constexpr int kSmV = kSmK + kKSlots * kKSlotBytes;        // V^T slots
constexpr int kSmScale = kSmV + kVSlots * kVSlotBytes;    // 2 slots: k'[128], vs[128]
constexpr int kSmRows = kSmScale + 2 * 1024;              // c[2][128], l[2][128], sp[2][128] floats (by unit parity)
constexpr int kSmStage = kSmRows + 6 * kRows * 4;         // epilogue: 4 x [32 rows][128 B]
constexpr int kSmBars = kSmStage + 4 * 4096;
// Barriers.  "Pair" barriers are waited on by the even CTA's MMA issuer and
// count arrivals from both CTAs (the odd CTA arrives through the cluster);
// "both" barriers are arrived on in both CTAs by one multicast MMA commit.
//
// Every K tile and V^T tile has one "full" barrier (by tile parity), so the
// MMA issuer waits once per operand per tile: a wait or a commit between two
// MMAs leaves the tensor pipe idle for tens of cycles, and the issuer's
// waits and commits add up on the critical path.  QK^T(t) done (S full) also
// frees the K slots of tile t.
enum : int {
  B_KFULL = 0,      // [2] by tile parity, pair: the tile's K landed in both CTAs
  B_VFULL = 2,      // [2] by tile parity, pair: the tile's V^T chunks landed in both CTAs
  B_VEMPTY = 4,     // [2] by tile parity, both: the tile's PV is done (V^T slots free)
  B_SCFULL = 6,     // [2] the tile's scales landed (each CTA loads its own copy)
  B_SCEMPTY = 8,    // [2] every softmax warp read them
  B_SFULL = 10,     // [2] both: S of a tile is in TMEM (and its K slots are free)
  B_PFULL = 12,     // [2] pair: P of a tile is in TMEM (every softmax warp of both CTAs)
  B_QFULL = 14,     // Q landed (in the even CTA: in both CTAs)
  B_QREADY = 15,    // this CTA's Q codes on the int8 grid are written
  B_QREADY2 = 16,   // pair: both CTAs' Q codes are written
  B_QEMPTY = 17,    // both: the unit's last QK^T is done
  B_OFULL = 18,     // both: the unit's last PV is done
  B_OEMPTY = 19,    // pair: the epilogue of both CTAs has read O
  B_STATS = 20,     // [2] by unit parity: the softmax's row sums are written
  B_STALL = 22,     // test hook: nothing arrives
  B_DRAIN = 23,     // both: every MMA is done
  B_QSOON = 24,     // the unit's Q may be prefetched
  kNumBars = 25
};
constexpr int kSmTmemSlot = kSmBars + kNumBars * 8;
constexpr int kAttnSmem = kSmTmemSlot + 16 + 1024;  // + alignment slack
static_assert(kAttnSmem <= 227 * 1024, "shared memory budget");

// The MMA issuer arrives on B_QSOON when it issues QK^T for the tile kQSoon
// tiles before its unit's last; the Q producer then prefetches the next
// unit's Q rows into L2, so that they are there when Q's slot frees up.
constexpr int kQSoon = 4;
constexpr float kLift = 6.f;   // a unit's first reference sits 2^kLift above its first tile's max
constexpr float kLazy = 14.f;  // the softmax reference moves when a row max grows by more than 2^kLazy;
                               // P' = p * v_scale * 2^-ev then stays below 2^14, inside the fp16 range

constexpr uint32_t kTmO = 0;
constexpr uint32_t kTmS = 256;
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
// V^T chunks of a tile of nb blocks.
__device__ __forceinline__ int n_chunks(int nb) { return (nb + 3) / 4; }

struct Ctx {
  uint32_t sbase;    // shared address of the aligned base
  uint32_t tb;       // TMEM base address (the same in both CTAs)
  uint32_t rank;     // 0: the even CTA of the pair (issues the MMAs), 1: the odd one
  int pair, n_pairs; // this pair's index and the number of pairs
  int u0, u1, ustep; // this pair's units: u0, u0 + ustep, ... below u1
  WaitCtl wc;
  __device__ uint32_t bar(int i) const { return sbase + kSmBars + 8 * i; }
  // Bounded wait.  Phases completed by the other CTA of the pair hand over
  // data that TMA copies or tcgen05 operations wrote (the copy's complete_tx,
  // the MMA commit, or tcgen05.wait + fence before the arrival order it), so
  // an acquire at CTA scope suffices; a cluster-scope acquire costs the MMA
  // issuer ~100 cycles more per wait.
  __device__ bool wait(int i, uint32_t parity, int site) const { return mbar_wait(bar(i), parity, wc, site); }
  // Bounded wait acquiring at cluster scope: for a phase that publishes the
  // other CTA's generic-proxy shared-memory writes (the int8 Q codes).
  __device__ bool wait_cluster(int i, uint32_t parity, int site) const {
    return mbar_wait_cluster(bar(i), parity, wc, site);
  }
  // The same by all 32 lanes of a warp with one outcome for the warp, so that
  // the warp-collective tcgen05.ld/st and __syncwarp that follow never see a
  // diverged warp, also when a wait runs out.
  __device__ bool warp_wait(int i, uint32_t parity, int site) const {
    return __all_sync(0xffffffffu, wait(i, parity, site));
  }
  // Arrive on a pair barrier (in the even CTA), publishing this thread's
  // generic-proxy writes to the other CTA.
  __device__ void arrive_pair(int i) const {
    if (rank == 0) mbar_arrive(bar(i));
    else mbar_arrive_cluster(cluster_addr(bar(i), 0));
  }
  // The same for a tensor-memory hand-off (the caller has waited for its
  // tcgen05.st/ld and fenced with tcgen05.fence::before_thread_sync).
  __device__ void arrive_pair_tmem(int i) const {
    if (rank == 0) mbar_arrive(bar(i));
    else mbar_arrive_remote(cluster_addr(bar(i), 0));
  }
};

// ------------------------------------------------------------------ producers
// A thread's TMA copies complete about one at a time (measured on GB300: one
// issuing thread moves ~29-36 B/clk of 16 KB tiles from L2 into shared memory
// whatever the number in flight, four threads ~70 B/clk), so every stream
// of copies is spread over several lanes, each with its own slots.
//
// Each CTA loads its own half of every K tile and V^T chunk into its own
// shared memory; both copies complete their bytes on the even CTA's barrier
// (the odd CTA's through the pair form of the TMA load), which expects both
// halves, so its phase means "both halves landed" to the MMA issuer.

// K: lane s loads region r = s % 4 (dims [64 r, 64 r + 64)) of the tiles of
// parity s / 4 into slot s: this CTA's N/2 keys of the tile, from key
// rank * N/2 on, N = 16 nb (the MMA takes N/2 rows from each CTA's slot).  The
// slot is free again once QK^T of the tile two before is done (S full).
__device__ __forceinline__ void role_producer_k(const AttnParams& p, const AttnMaps& m, const Ctx& c, int s) {
  const int r = s & 3, par = s >> 2;
  uint32_t uses = 0, tc = 0;  // tiles this slot held; tiles so far
  bool ok = true;
  for (int u = c.u0; u < c.u1 && ok; u += c.ustep) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const UnitGeom ug = unit_geom(un.t0, 2 * p.TQ, sg, p.S, p.W);
    for (int j = 0; j < ug.n_tiles; ++j) {
      if ((int)((tc + j) & 1) != par) continue;
      const TileGeom tg = tile_geom(ug, j, p.S, p.W);
      const int row = logical_block_row(sg, tg.kb0) + (int)c.rank * tg.nb * (kPage / 2);
      if (!(ok = c.wait(B_SFULL + par, (uses & 1) ^ 1, 10))) break;
      const uint32_t fb = c.bar(B_KFULL + par);
      if (c.rank == 0) {
        mbar_expect_tx(fb, 2 * kKSlotBytes);  // one of four arrivals: this region of both CTAs
        tma_load_3d(c.sbase + kSmK + s * kKSlotBytes, &m.k, fb, r * 64, row, un.g);
      } else {
        tma_load_3d_pair(c.sbase + kSmK + s * kKSlotBytes, &m.k, cluster_addr(fb, 0), r * 64, row, un.g);
      }
      ++uses;
    }
    tc += ug.n_tiles;
  }
  // every issued copy lands before the CTA may exit: the MMAs that read the
  // slot's last copy are done (bounded: on an error they may never run)
  if (uses > 0) (void)mbar_wait_drain(c.bar(B_SFULL + par), (uses - 1) & 1, kDrainNs);
}

// V^T: lane s loads chunk ch = s % 2 (keys [64 ch, 64 ch + 64)) of the tiles of
// parity s / 2 into slot s: this CTA's 128 of the 256 dims.  Lane (parity, 0)
// of the even CTA expects the bytes of all the tile's chunks in both CTAs;
// the slot is free again once PV of the tile two before is done.
__device__ __forceinline__ void role_producer_v(const AttnParams& p, const AttnMaps& m, const Ctx& c, int s) {
  const int ch = s & 1, par = s >> 1;
  uint32_t uses = 0, tc = 0;  // tiles of this parity so far; tiles so far
  bool ok = true;
  for (int u = c.u0; u < c.u1 && ok; u += c.ustep) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const UnitGeom ug = unit_geom(un.t0, 2 * p.TQ, sg, p.S, p.W);
    for (int j = 0; j < ug.n_tiles; ++j) {
      if ((int)((tc + j) & 1) != par) continue;
      const int nch = n_chunks(tile_width(ug, j));
      const uint32_t use = uses++;
      // every lane waits for every tile of its parity, also one it has no
      // chunk of: a parity wait cannot tell phase k from k - 2, so a lane that
      // skipped a wait could pass the next one two phases early
      if (!(ok = c.wait(B_VEMPTY + par, (use & 1) ^ 1, 11))) break;
      if (ch >= nch) continue;  // a tile of one chunk
      const int crow = logical_block_row(sg, tile_geom(ug, j, p.S, p.W).kb0);
      const uint32_t fb = c.bar(B_VFULL + par);
      const uint32_t dst = c.sbase + kSmV + s * kVSlotBytes;
      if (c.rank == 0) {
        if (ch == 0) mbar_expect_tx(fb, (uint32_t)nch * 2 * kVSlotBytes);
        tma_load_3d(dst, &m.v, fb, crow + ch * kChunkKeys, 0, un.g);
      } else {
        tma_load_3d_pair(dst, &m.v, cluster_addr(fb, 0), crow + ch * kChunkKeys, kHeadDim / 2, un.g);
      }
    }
    tc += ug.n_tiles;
  }
  if (uses > 0) (void)mbar_wait_drain(c.bar(B_VEMPTY + par), (uses - 1) & 1, kDrainNs);
}

// Prefetch into L2 the rows of TQ tokens from t0 in a [tokens][HQ][256] bf16
// tensor (q or the output gate): per token its G heads are contiguous.
__device__ __forceinline__ void prefetch_rows(const AttnParams& p, const __nv_bfloat16* base, int t0, int g,
                                              const SeqGeom& sg) {
  const int tok0 = sg.q_off + (t0 - sg.q_start);
  for (int i = 0; i < p.TQ; ++i) {
    const int tok = tok0 + i;
    if (tok >= sg.q_off && tok < sg.q_off + sg.n_q)
      bulk_prefetch_l2(base + ((size_t)tok * p.HQ + (size_t)g * p.G) * kHeadDim, (uint32_t)p.G * kHeadDim * 2);
  }
}

// Q of each unit (this CTA's 128 rows, after the pair's last QK^T of the
// previous unit): lane r < 4 loads region r.  Lane 0 also prefetches into L2
// the unit's Q rows and the previous unit's output-gate rows (both a few tiles
// before they are needed) and, in the odd CTA, passes the arrival of its Q on
// to the even CTA.  Lane 4 loads the K/V scales of each tile (two-slot ring
// by tile parity).
__device__ __forceinline__ void role_producer_q(const AttnParams& p, const AttnMaps& m, const Ctx& c, int r) {
  uint32_t ts = 0;  // tiles whose scales were loaded
  int k_unit = 0;   // units whose Q was loaded
  bool ok = true;
  int prev_t0 = 0, prev_g = 0;
  SeqGeom prev_sg{};
  // rows still on their way in from another stream: wait for their flag
  if (r < 4 && p.q_ready && c.u0 < c.u1) ok = flag_wait(p.q_ready, p.q_epoch, c.wc, 18);
  for (int u = c.u0; u < c.u1 && ok; u += c.ustep) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const int t0 = un.t0 + (int)c.rank * p.TQ;  // this CTA's first token
    if (r == 4) {
      const UnitGeom ug = unit_geom(un.t0, 2 * p.TQ, sg, p.S, p.W);
      for (int j = 0; j < ug.n_tiles; ++j) {
        const uint32_t s = ts & 1;
        if (!(ok = c.wait(B_SCEMPTY + s, ((ts >> 1) & 1) ^ 1, 14))) break;
        const TileGeom tg = tile_geom(ug, j, p.S, p.W);
        const int crow = logical_block_row(sg, tg.kb0);
        const uint32_t bytes = (uint32_t)(tg.nb * kPage * 4);
        const uint32_t fb = c.bar(B_SCFULL + s);
        mbar_expect_tx(fb, 2 * bytes);
        bulk_load(c.sbase + kSmScale + s * 1024, p.ks + (size_t)un.g * p.n_tok_cap + crow, bytes, fb);
        bulk_load(c.sbase + kSmScale + s * 1024 + 512, p.vs + (size_t)un.g * p.n_tok_cap + crow, bytes, fb);
        ++ts;
      }
      continue;
    }
    // q row (token position in q) of this CTA's first token; negative or past
    // the sequence where the unit overhangs it: those rows are never output
    const int tok0 = sg.q_off + (t0 - sg.q_start);
    if (k_unit > 0) {
      if (!(ok = c.wait(B_QSOON, (k_unit - 1) & 1, 12))) break;
      if (r == 0) {
        prefetch_rows(p, p.q, t0, un.g, sg);
        if (p.gate) prefetch_rows(p, p.gate, prev_t0, prev_g, prev_sg);
      }
      if (!(ok = c.wait(B_QEMPTY, (k_unit - 1) & 1, 13))) break;
    }
    prev_t0 = t0;
    prev_g = un.g;
    prev_sg = sg;
    mbar_expect_tx(c.bar(B_QFULL), kRegionBytes);
    tma_load_3d(c.sbase + kSmQ + r * kRegionBytes, &m.q, c.bar(B_QFULL), r * 64, un.g * p.G, tok0);
    if (c.rank == 1 && r == 0) {
      if (!(ok = c.wait(B_QFULL, k_unit & 1, 17))) break;
      mbar_arrive_cluster(cluster_addr(c.bar(B_QFULL), 0));
    }
    ++k_unit;
  }
  if (r < 4 && k_unit > 0) (void)mbar_wait_drain(c.bar(B_QFULL), (k_unit - 1) & 1, kDrainNs);
  for (uint32_t i = 0; i < 2; ++i)
    if (ts > i) (void)mbar_wait_drain(c.bar(B_SCFULL + ((ts - 1 - i) & 1)), ((ts - 1 - i) >> 1) & 1, kDrainNs);
}

// ------------------------------------------------------------------ MMA issuer
// One thread of the even CTA issues every MMA of the pair: 256 query rows
// (128 in each CTA's TMEM lanes) against the tile's keys.
//
// This thread is the pipeline's critical path (clock64 stamps on GB300): each
// tcgen05.mma costs it ~70-80 cycles to issue whatever its operands, and a
// wait, a commit or a branch between MMA groups ~60-150, while the tensor pipe
// runs a tile's 16 QK^T MMAs in ~1024 cycles and its 8 PV MMAs in ~1024.  So
// the MMAs of a tile are issued from one asm block each and the rare arrivals
// and commits are predicated or kept off the common path.

// S(t) = Q K(t)^T for a tile: 16 MMAs, Q region r at qd + 1024 r and the K
// slot's region r at kd + 512 r (start addresses in 16-byte units), k-step q
// at + 2 q within the 128-byte swizzled rows; the first MMA overwrites D.
static_assert(kRegionBytes / 16 == 1024 && kKSlotBytes / 16 == 512, "descriptor steps of mma_qk_tile");
__device__ __forceinline__ void mma_qk_tile(uint32_t d, uint64_t qd, uint64_t kd, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .b64 a, b;\n\t.reg .pred pf, pt;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      "add.s64 a, %1, 2;\n\tadd.s64 b, %2, 2;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 4;\n\tadd.s64 b, %2, 4;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 6;\n\tadd.s64 b, %2, 6;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 1024;\n\tadd.s64 b, %2, 512;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 1026;\n\tadd.s64 b, %2, 514;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 1028;\n\tadd.s64 b, %2, 516;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 1030;\n\tadd.s64 b, %2, 518;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 2048;\n\tadd.s64 b, %2, 1024;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 2050;\n\tadd.s64 b, %2, 1026;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 2052;\n\tadd.s64 b, %2, 1028;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 2054;\n\tadd.s64 b, %2, 1030;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 3072;\n\tadd.s64 b, %2, 1536;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 3074;\n\tadd.s64 b, %2, 1538;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 3076;\n\tadd.s64 b, %2, 1540;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 3078;\n\tadd.s64 b, %2, 1542;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "}" ::"r"(d), "l"(qd), "l"(kd), "r"(idesc), "r"(0u)
      : "memory");
}
// O (+)= P' V for a full tile: 8 MMAs, P' of 64-key chunk ch at TMEM column
// a + 64 ch + 8 ks, its V^T slot at vd0 / vd1 + 2 ks; the first MMA
// accumulates iff acc0.
static_assert(kChunkKeys == 64 && kTileKeys == 2 * kChunkKeys, "TMEM column steps of mma_pv_tile");
__device__ __forceinline__ void mma_pv_tile(uint32_t d, uint32_t a, uint64_t vd0, uint64_t vd1, uint32_t idesc,
                                            uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .b64 b;\n\t.reg .b32 ta;\n\t.reg .pred pa, pt;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\tsetp.eq.b32 pt, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %4, pa;\n\t"
      "add.u32 ta, %1, 8;\n\tadd.s64 b, %2, 2;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], b, %4, pt;\n\t"
      "add.u32 ta, %1, 16;\n\tadd.s64 b, %2, 4;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], b, %4, pt;\n\t"
      "add.u32 ta, %1, 24;\n\tadd.s64 b, %2, 6;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], b, %4, pt;\n\t"
      "add.u32 ta, %1, 64;\n\tadd.s64 b, %3, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], b, %4, pt;\n\t"
      "add.u32 ta, %1, 72;\n\tadd.s64 b, %3, 2;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], b, %4, pt;\n\t"
      "add.u32 ta, %1, 80;\n\tadd.s64 b, %3, 4;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], b, %4, pt;\n\t"
      "add.u32 ta, %1, 88;\n\tadd.s64 b, %3, 6;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], b, %4, pt;\n\t"
      "}" ::"r"(d), "r"(a), "l"(vd0), "l"(vd1), "r"(idesc), "r"(acc0), "r"(0u)
      : "memory");
}
// mma_commit_pair when `pred` holds, without a branch.
__device__ __forceinline__ void mma_commit_pair_if(uint32_t bar, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
      "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
      "h"((uint16_t)3), "r"((uint32_t)pred)
      : "memory");
}

__device__ __forceinline__ void role_mma(const AttnParams& p, const Ctx& c) {
  uint32_t tc = 0;  // global tile counter: K/V slots and S buffer by its parity
  int k_unit = 0;
  bool ok = true;
  const uint32_t id_pv = idesc_f16(kUnitRows, kHeadDim, false, false);
  const uint32_t qsoon_peer = cluster_addr(c.bar(B_QSOON), 1);
  const uint64_t qd = sdesc_k_sw128(c.sbase + kSmQ);
  // K slots and V^T slots by tile parity (selected, not indexed: kept in registers)
  const uint64_t kd0 = sdesc_k_sw128(c.sbase + kSmK), kd1 = sdesc_k_sw128(c.sbase + kSmK + 4 * kKSlotBytes);
  const uint64_t vd00 = sdesc_k_sw128(c.sbase + kSmV), vd01 = sdesc_k_sw128(c.sbase + kSmV + kVSlotBytes);
  const uint64_t vd10 = sdesc_k_sw128(c.sbase + kSmV + 2 * kVSlotBytes);
  const uint64_t vd11 = sdesc_k_sw128(c.sbase + kSmV + 3 * kVSlotBytes);
  for (int u = c.u0; u < c.u1 && ok; u += c.ustep, ++k_unit) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const UnitGeom ug = unit_geom(un.t0, 2 * p.TQ, sg, p.S, p.W);
    const int n = ug.n_tiles;
    const int jsoon = imax(0, n - kQSoon);  // its QK^T lets the next unit's Q rows be prefetched
    const int qbar = p.debug_stall ? B_STALL : (p.q_mode == 1 ? B_QREADY2 : B_QFULL);
    if (!(ok = (qbar == B_QREADY2 ? c.wait_cluster(qbar, k_unit & 1, 20) : c.wait(qbar, k_unit & 1, 20)))) break;
    // S(j) = Q K(j)^T, then the unit's rare arrivals: Q free after its last
    // QK^T, the prefetch of the next unit's Q rows a few tiles before
    auto qk = [&](int j) {
      const uint32_t t = tc + j;
      const uint32_t d = c.tb + kTmS + (t & 1) * kTileKeys;
      const uint32_t id = idesc_f16(kUnitRows, tile_width(ug, j) * kPage, true, true);  // bf16 Q, bf16 K codes
      if (!c.wait(B_KFULL + (t & 1), (t >> 1) & 1, 21)) return false;
      tc_fence_after();
      mma_qk_tile(d, qd, (t & 1) ? kd1 : kd0, id);
      mma_commit_pair(c.bar(B_SFULL + (t & 1)));  // S(t) ready; tile t's K slots free
      mma_commit_pair_if(c.bar(B_QEMPTY), j == n - 1);
      if (__builtin_expect(j == jsoon, 0)) {
        // a timing hint, no data: the CTA-scope arrive (a cluster-scope
        // release would wait for this thread's MMAs in flight)
        mbar_arrive(c.bar(B_QSOON));
        mbar_arrive_remote(qsoon_peer);
      }
      return true;
    };
    // O (+)= P(j) V(j), then O's release to the epilogue after the unit's last
    auto pv = [&](int j) {
      const uint32_t t = tc + j;
      if (!c.wait(B_VFULL + (t & 1), (t >> 1) & 1, 23)) return false;
      if (!c.wait(B_PFULL + (t & 1), (t >> 1) & 1, 22)) return false;
      // the previous unit's O was read by the epilogue of both CTAs
      if (__builtin_expect(j == 0 && k_unit > 0, 0) && !c.wait(B_OEMPTY, (k_unit - 1) & 1, 24)) return false;
      const uint32_t a = c.tb + kTmS + (t & 1) * kTileKeys;
      const int nb = tile_width(ug, j);
      const uint32_t acc0 = j > 0 ? 1u : 0u;
      const uint64_t vd0 = (t & 1) ? vd10 : vd00, vd1 = (t & 1) ? vd11 : vd01;
      tc_fence_after();
      // k-step ks of chunk ch covers keys [64 ch + 16 ks, +16); P' of chunk ch
      // sits at S columns [64 ch, 64 ch + 32)
      if (__builtin_expect(nb == kTileBlocks, 1)) {
        mma_pv_tile(c.tb + kTmO, a, vd0, vd1, id_pv, acc0);
      } else {
        for (int ch = 0; ch < n_chunks(nb); ++ch) {
          const int nks = imin(4, nb - 4 * ch);
          for (int ks = 0; ks < nks; ++ks)
            mma_ts_pair(c.tb + kTmO, a + 64 * ch + 8 * ks, (ch ? vd1 : vd0) + (uint64_t)(2 * ks), id_pv,
                        (ch > 0 || ks > 0) ? 1u : acc0);
        }
      }
      mma_commit_pair(c.bar(B_VEMPTY + (t & 1)));  // tile t's V^T slots free; O holds PV up to tile t
      mma_commit_pair_if(c.bar(B_OFULL), j == n - 1);
      return true;
    };
    // QK^T(j) before PV(j - 1): the tensor pipe computes the next scores
    // while the softmax handles the current ones
    if (!(ok = qk(0))) break;
    for (int j = 1; j < n; ++j) {
      if (__builtin_expect(!qk(j), 0) || __builtin_expect(!pv(j - 1), 0)) {
        ok = false;
        break;
      }
    }
    if (!ok || !(ok = pv(n - 1))) break;
    tc += n;
  }
  // every issued MMA completes before TMEM is freed (the odd CTA waits for
  // its copy of this arrival too)
  mma_commit_pair(c.bar(B_DRAIN));
  (void)mbar_wait_drain(c.bar(B_DRAIN), 0, kDrainNs);
}

// ------------------------------------------------------------------ softmax
// Two warps per TMEM lane quadrant, each owning 16 whole rows of the
// quadrant's 32 (lanes 32 qd + 16 hh + [0, 16)) across all 128 key columns of
// a tile, read and written in the 16-lane TMEM shapes: thread t holds rows
// t/4 and t/4 + 8 of the 16 and, of every 8 key columns, columns 2 (t % 4)
// and 2 (t % 4) + 1.  Each K/V scale a thread loads so serves two rows (the
// scale loads, broadcast from shared memory, bound the softmax otherwise), and
// a row's maximum and sum take two shuffles among the four threads that share
// it, with no exchange between warps.  Each CTA of a pair runs its own
// softmax over its own 128 rows; only the arrival that releases PV goes to the
// even CTA, whose MMA issuer multiplies both.
__device__ __forceinline__ void role_softmax(const AttnParams& p, const Ctx& c, uint8_t* sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lb = 32 * (warp & 3) + 16 * ((warp - 4) >> 2);  // first of this warp's 16 rows (TMEM lanes)
  const int tcol = 2 * (lane & 3);                          // this thread's first column of every 8
  const int rr[2] = {lb + (lane >> 2), lb + (lane >> 2) + 8};  // its two rows
  const uint32_t lane_off = (uint32_t)lb << 16;
  float* c_rows = reinterpret_cast<float*>(sm + kSmRows);
  float* l_rows = c_rows + 2 * kRows;   // [unit parity][row]
  float* sp_rows = c_rows + 4 * kRows;  // [unit parity][row]
  const bool u8 = p.p_mode == 1;
  uint32_t tc = 0;
  int k_unit = 0;
  bool ok = true;
  for (int u = c.u0; u < c.u1 && ok; u += c.ustep, ++k_unit) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    const UnitGeom ug = unit_geom(un.t0, 2 * p.TQ, sg, p.S, p.W);
    const int n = ug.n_tiles;
    const int t0 = un.t0 + (int)c.rank * p.TQ;  // this CTA's first token
    const int t_row[2] = {t0 + rr[0] / p.G, t0 + rr[1] / p.G};
    const float ev = (float)pow2_ceil_exp(__uint_as_float(p.vsmax[un.seq * p.HKV + un.g]));
    // the per-row query scale (s_q on the int8 grid, 1 for the bf16 query;
    // sm_scale * log2(e) is in the K scales), kept positive so that -inf
    // scores stay -inf
    float c_row[2] = {1.f, 1.f};
    if (p.q_mode == 1) {
      if (!(ok = c.warp_wait(B_QREADY, k_unit & 1, 30))) break;
      c_row[0] = c_rows[(k_unit & 1) * kRows + rr[0]];
      c_row[1] = c_rows[(k_unit & 1) * kRows + rr[1]];
    }
    c_row[0] = fmaxf(c_row[0], 1e-30f);
    c_row[1] = fmaxf(c_row[1], 1e-30f);
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f}, sp_prev[2] = {1.f, 1.f};
    for (int j = 0; j < n; ++j) {
      const uint32_t t = tc + j;
      const TileGeom tg = tile_geom(ug, j, p.S, p.W);
      if (!(ok = c.warp_wait(B_SFULL + (t & 1), (t >> 1) & 1, 31))) break;
      const uint32_t sd = c.tb + lane_off + kTmS + (t & 1) * kTileKeys;
      // this thread's K scales at +8k (two floats each); its V scales 128 floats on
      const float* ksp = reinterpret_cast<const float*>(sm + kSmScale + (t & 1) * 1024) + tcol;
      const float* vsp = ksp + 128;
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_16x256b_x16(sd, sv);
      // the tile's scales (normally there long since), checked while the
      // score load is in flight
      const bool oks = c.warp_wait(B_SCFULL + (t & 1), (t >> 1) & 1, 32);
      tmem_wait_ld(sv);
      if (!(ok = oks)) break;
      // y = S * k_scale (masked: -inf), in place, and each row's maximum; the
      // products in fp32 pairs, the maximum three operands at a time
      // A tile every row sees in full (most of them) takes a loop without the
      // mask: with the mask's selects inside one loop under a condition, they
      // were executed as predicated instructions on every tile.
      const bool full = !tg.needs_mask && tg.nb == kTileBlocks;
      float mx[2][2] = {{-INFINITY, -INFINITY}, {-INFINITY, -INFINITY}};
      if (full) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 k2 = *reinterpret_cast<const float2*>(ksp + 8 * k);
          const float2 a = mul2(make_float2(__uint_as_float(sv[4 * k]), __uint_as_float(sv[4 * k + 1])), k2);
          const float2 b = mul2(make_float2(__uint_as_float(sv[4 * k + 2]), __uint_as_float(sv[4 * k + 3])), k2);
          sv[4 * k] = __float_as_uint(a.x);
          sv[4 * k + 1] = __float_as_uint(a.y);
          sv[4 * k + 2] = __float_as_uint(b.x);
          sv[4 * k + 3] = __float_as_uint(b.y);
          mx[0][k & 1] = max3(mx[0][k & 1], a.x, a.y);
          mx[1][k & 1] = max3(mx[1][k & 1], b.x, b.y);
        }
      } else {
        unsigned long long vis[2][2];  // [row][key half] >> tcol
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) vis[i][hf] = visible_columns(tg, t_row[i], p.S, p.W, hf) >> tcol;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 k2 = *reinterpret_cast<const float2*>(ksp + 8 * k);
          float2 a = mul2(make_float2(__uint_as_float(sv[4 * k]), __uint_as_float(sv[4 * k + 1])), k2);
          float2 b = mul2(make_float2(__uint_as_float(sv[4 * k + 2]), __uint_as_float(sv[4 * k + 3])), k2);
          const int hf = k >> 3, sh = 8 * (k & 7);
          a.x = ((vis[0][hf] >> sh) & 1ull) ? a.x : -INFINITY;
          a.y = ((vis[0][hf] >> (sh + 1)) & 1ull) ? a.y : -INFINITY;
          b.x = ((vis[1][hf] >> sh) & 1ull) ? b.x : -INFINITY;
          b.y = ((vis[1][hf] >> (sh + 1)) & 1ull) ? b.y : -INFINITY;
          sv[4 * k] = __float_as_uint(a.x);
          sv[4 * k + 1] = __float_as_uint(a.y);
          sv[4 * k + 2] = __float_as_uint(b.x);
          sv[4 * k + 3] = __float_as_uint(b.y);
          mx[0][k & 1] = max3(mx[0][k & 1], a.x, a.y);
          mx[1][k & 1] = max3(mx[1][k & 1], b.x, b.y);
        }
      }
      // the reference of a row moves only when its max grew by more than 2^kLazy
      float alpha[2] = {1.f, 1.f}, mref[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float m = fmaxf(mx[i][0], mx[i][1]);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const float my = m * c_row[i];  // log2 units
        if (m_run[i] == -INFINITY) {
          m_run[i] = my == -INFINITY ? my : my + kLift;  // alpha irrelevant: nothing accumulated yet
          alpha[i] = 0.f;
        } else if (my > m_run[i] + kLazy) {
          alpha[i] = ex2_approx(m_run[i] - my);
          m_run[i] = my;
        }
        mref[i] = m_run[i] == -INFINITY ? 0.f : m_run[i] + ev;
      }
      // p = 2^(y c - mref); P' = p * v_scale (V scale folded into P)
      float2 s2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      const float2 c2[2] = {make_float2(c_row[0], c_row[0]), make_float2(c_row[1], c_row[1])};
      const float2 nm2[2] = {make_float2(-mref[0], -mref[0]), make_float2(-mref[1], -mref[1])};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 v2 = *reinterpret_cast<const float2*>(vsp + 8 * k);
        const float2 a = fma2(make_float2(__uint_as_float(sv[4 * k]), __uint_as_float(sv[4 * k + 1])), c2[0], nm2[0]);
        const float2 b = fma2(make_float2(__uint_as_float(sv[4 * k + 2]), __uint_as_float(sv[4 * k + 3])), c2[1], nm2[1]);
        const float2 pa = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        const float2 pb = make_float2(ex2_approx(b.x), ex2_approx(b.y));
        s2[0] = add2(s2[0], pa);
        s2[1] = add2(s2[1], pb);
        const float2 wa = mul2(pa, v2), wb = mul2(pb, v2);
        sv[4 * k] = __float_as_uint(wa.x);
        sv[4 * k + 1] = __float_as_uint(wa.y);
        sv[4 * k + 2] = __float_as_uint(wb.x);
        sv[4 * k + 3] = __float_as_uint(wb.y);
      }
      // this warp is done with the tile's scales
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(B_SCEMPTY + (t & 1)));
      float corr[2] = {alpha[0], alpha[1]};
#pragma unroll
      for (int i = 0; i < 2; ++i) l_run[i] = l_run[i] * alpha[i] + (s2[i].x + s2[i].y);
      if (u8) {  // P' per row on the u8 grid over the whole tile, scale max/255
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float pm = 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) pm = max3(pm, __uint_as_float(sv[4 * k + 2 * i]), __uint_as_float(sv[4 * k + 2 * i + 1]));
          pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
          pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
          const float sp = pm > 0.f ? __fdiv_rn(pm, 255.f) : sp_prev[i];
          const float inv = pm > 0.f ? __fdiv_rn(255.f, pm) : 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            sv[4 * k + 2 * i] = __float_as_uint(rintf(__uint_as_float(sv[4 * k + 2 * i]) * inv));
            sv[4 * k + 2 * i + 1] = __float_as_uint(rintf(__uint_as_float(sv[4 * k + 2 * i + 1]) * inv));
          }
          corr[i] = alpha[i] * __fdiv_rn(sp_prev[i], sp);
          sp_prev[i] = sp;
        }
      }
      // P' as fp16 pairs over S columns [0, 32) (keys 0-63) and [64, 96) (keys
      // 64-127), where the PV issuer reads them
      uint32_t pk0[16], pk1[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        pk0[2 * k] = pack_half2(__uint_as_float(sv[4 * k]), __uint_as_float(sv[4 * k + 1]));
        pk0[2 * k + 1] = pack_half2(__uint_as_float(sv[4 * k + 2]), __uint_as_float(sv[4 * k + 3]));
        pk1[2 * k] = pack_half2(__uint_as_float(sv[32 + 4 * k]), __uint_as_float(sv[32 + 4 * k + 1]));
        pk1[2 * k + 1] = pack_half2(__uint_as_float(sv[32 + 4 * k + 2]), __uint_as_float(sv[32 + 4 * k + 3]));
      }
      tmem_st_16x128b_x8(sd, pk0);
      tmem_st_16x128b_x8(sd + 64, pk1);
      // O holds PV up to tile j-1 once that MMA is done; rescale this warp's
      // rows in place.  A wait that runs out skips the rescale (the error word
      // is set; the results of the call are void).
      if (j > 0 && __any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f) &&
          c.warp_wait(B_VEMPTY + ((t - 1) & 1), ((t - 1) >> 1) & 1, 33)) {
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          const uint32_t oa = c.tb + lane_off + kTmO + 64 * cc;
          tmem_ld_16x256b_x8(oa, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 x = mul2(make_float2(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1])),
                                  make_float2(corr[0], corr[0]));
            const float2 y = mul2(make_float2(__uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3])),
                                  make_float2(corr[1], corr[1]));
            o[4 * k] = __float_as_uint(x.x);
            o[4 * k + 1] = __float_as_uint(x.y);
            o[4 * k + 2] = __float_as_uint(y.x);
            o[4 * k + 3] = __float_as_uint(y.y);
          }
          tmem_st_16x256b_x8(oa, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) c.arrive_pair_tmem(B_PFULL + (t & 1));
    }
    if (!ok) break;
    tc += n;
    // each row's sum over the four threads that share it
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float l = l_run[i];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if ((lane & 3) == 0) {
        l_rows[(k_unit & 1) * kRows + rr[i]] = l;
        sp_rows[(k_unit & 1) * kRows + rr[i]] = sp_prev[i];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(B_STATS + (k_unit & 1)));
  }
  tmem_wait_st();
}

// ------------------------------------------------------------------ Q codes / epilogue
struct RowInfo {
  bool valid;
  size_t off;  // element offset of the row in q / out
};

// Row r of the CTA whose first token is t0, kv head g.
__device__ __forceinline__ RowInfo row_info(const AttnParams& p, int t0, int g, const SeqGeom& sg, int r) {
  RowInfo ri;
  const int t_row = t0 + r / p.G;
  const int h_row = g * p.G + r % p.G;
  ri.valid = t_row >= sg.q_start && t_row < sg.q_start + sg.n_q;
  ri.off = ri.valid ? ((size_t)(sg.q_off + t_row - sg.q_start) * p.HQ + h_row) * kHeadDim : 0;
  return ri;
}

// 16-byte piece `piece` of row `row` of a tile of 128-byte rows written by TMA
// with the 128-byte swizzle (1024-byte aligned): the pieces of a row are
// permuted by the row's index mod 8.  The epilogue stage uses the same layout,
// which makes both a thread per row and four rows per warp instruction free of
// bank conflicts.
__device__ __forceinline__ uint4* swz(uint8_t* base, int row, int piece) {
  return reinterpret_cast<uint4*>(base + row * 128 + ((piece ^ (row & 7)) << 4));
}

// The rows lane `lane` moves in the four-rows-per-instruction pattern:
// row 4k + lane/8 of the warp's 32, k = 0..7.
struct LaneRows {
  uint32_t row[8];  // row index in q / out (element offset row * 256)
  uint32_t valid;   // bit k: row k is a query row of the call
};
__device__ __forceinline__ LaneRows lane_rows(const AttnParams& p, int t0, int g, const SeqGeom& sg, int qd,
                                              int lane) {
  LaneRows lr;
  lr.valid = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const RowInfo ri = row_info(p, t0, g, sg, 32 * qd + 4 * k + (lane >> 3));
    lr.row[k] = (uint32_t)(ri.off / kHeadDim);
    lr.valid |= (ri.valid ? 1u : 0u) << k;
  }
  return lr;
}

// Q on the pages' int8 grid (step a1), in place in shared memory: the row's
// codes rint(q * 127/absmax) clamped to [-127, 127], held exactly as bf16;
// returns s_q = absmax / 127 (sm_scale * log2(e) is in the K scales).
__device__ __forceinline__ float q_codes_int8(uint8_t* qs, int r) {
  float absmax = 0.f;
#pragma unroll 1
  for (int reg = 0; reg < 4; ++reg)
#pragma unroll
    for (int pc = 0; pc < 8; ++pc) {
      const uint4 v = *swz(qs + reg * kRegionBytes, r, pc);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        absmax = fmaxf(absmax, fabsf(__uint_as_float(w[e] << 16)));
        absmax = fmaxf(absmax, fabsf(__uint_as_float(w[e] & 0xffff0000u)));
      }
    }
  const float mul = absmax > 0.f ? __fdiv_rn(127.f, absmax) : 0.f;
#pragma unroll 1
  for (int reg = 0; reg < 4; ++reg)
#pragma unroll
    for (int pc = 0; pc < 8; ++pc) {
      uint4* a = swz(qs + reg * kRegionBytes, r, pc);
      const uint4 v = *a;
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = fminf(127.f, fmaxf(-127.f, rintf(__uint_as_float(w[e] << 16) * mul)));
        const float hi = fminf(127.f, fmaxf(-127.f, rintf(__uint_as_float(w[e] & 0xffff0000u) * mul)));
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        w[e] = *reinterpret_cast<uint32_t*>(&b);
      }
      *a = make_uint4(w[0], w[1], w[2], w[3]);
    }
  return __fdiv_rn(absmax, 127.f);
}

// Eight bf16 outputs times sigmoid of their eight bf16 gate values, rounded
// to bf16 again (the output gate, applied to the rounded attention output as
// a separate elementwise kernel would).
__device__ __forceinline__ uint4 gate8(uint4 v, uint4 g) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float lo = __uint_as_float(w[e] << 16) * __fdividef(1.f, 1.f + __expf(-__uint_as_float(gw[e] << 16)));
    const float hi =
        __uint_as_float(w[e] & 0xffff0000u) * __fdividef(1.f, 1.f + __expf(-__uint_as_float(gw[e] & 0xffff0000u)));
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    w[e] = *reinterpret_cast<uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// out = O / l (x s_p on the u8 grid) -> bf16 (step a8), 64 columns per round,
// times sigmoid(gate) when the call has an output gate.  O may be overwritten
// once the last round's TMEM loads are done, so the MMA issuer is released
// before the last stores.
__device__ __forceinline__ bool epilogue(const AttnParams& p, const Ctx& c, const LaneRows& lr, int k_unit,
                                         uint32_t to, const float* l_rows, const float* sp_rows, int r,
                                         uint8_t* stage, int lane) {
  if (!c.warp_wait(B_OFULL, k_unit & 1, 41)) return false;
  if (!c.warp_wait(B_STATS + (k_unit & 1), (k_unit >> 1) & 1, 42)) return false;
  tc_fence_after();
  const float l = l_rows[(k_unit & 1) * kRows + r];
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
      if (lane == 0) c.arrive_pair_tmem(B_OEMPTY);
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
    for (int pp = 0; pp < 8; ++pp) *swz(stage, lane, pp) = make_uint4(w[4 * pp], w[4 * pp + 1], w[4 * pp + 2], w[4 * pp + 3]);
    __syncwarp();
    if (p.gate) {
      uint4 g[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        g[k] = (lr.valid >> k) & 1u ? __ldg(reinterpret_cast<const uint4*>(p.gate + (size_t)lr.row[k] * kHeadDim + cb * 64) + pc)
                                    : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if ((lr.valid >> k) & 1u)
          *(reinterpret_cast<uint4*>(p.out + (size_t)lr.row[k] * kHeadDim + cb * 64) + pc) =
              gate8(*swz(stage, 4 * k + (lane >> 3), pc), g[k]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if ((lr.valid >> k) & 1u)
          *(reinterpret_cast<uint4*>(p.out + (size_t)lr.row[k] * kHeadDim + cb * 64) + pc) =
              *swz(stage, 4 * k + (lane >> 3), pc);
    }
  }
  return true;
}

__device__ __forceinline__ void role_correction(const AttnParams& p, const Ctx& c, uint8_t* sm) {
  const int r = threadIdx.x - 32 * (4 + kSoftmaxWarps);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3;
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  uint8_t* stage = sm + kSmStage + qd * 4096;
  float* c_rows = reinterpret_cast<float*>(sm + kSmRows);
  const float* l_rows = c_rows + 2 * kRows;
  const float* sp_rows = c_rows + 4 * kRows;
  int k_unit = 0;
  bool ok = true;
  int prev_t0 = 0, prev_g = 0;
  SeqGeom prev_sg{};
  for (int u = c.u0; u < c.u1 && ok; u += c.ustep, ++k_unit) {
    const Unit un = p.units[u];
    const SeqGeom sg = p.seqs[un.seq];
    if (p.q_mode == 1) {  // the unit's Q codes, in place, before the MMA may read Q
      if (!(ok = c.warp_wait(B_QFULL, k_unit & 1, 40))) break;
      c_rows[(k_unit & 1) * kRows + r] = q_codes_int8(sm + kSmQ, r);
      fence_proxy_async_shared();  // generic-proxy writes, read next by the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(c.bar(B_QREADY));
        c.arrive_pair(B_QREADY2);
      }
    }
    if (k_unit > 0)
      ok = epilogue(p, c, lane_rows(p, prev_t0, prev_g, prev_sg, qd, lane), k_unit - 1, c.tb + lane_off + kTmO,
                    l_rows, sp_rows, r, stage, lane);
    prev_t0 = un.t0 + (int)c.rank * p.TQ;
    prev_g = un.g;
    prev_sg = sg;
  }
  if (ok && k_unit > 0)
    (void)epilogue(p, c, lane_rows(p, prev_t0, prev_g, prev_sg, qd, lane), k_unit - 1, c.tb + lane_off + kTmO,
                   l_rows, sp_rows, r, stage, lane);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ AttnMaps m) {
  extern __shared__ uint8_t smraw[];
  // 1024-byte aligned base by pointer arithmetic on the shared array, so the
  // compiler keeps every access through `sm` in the shared address space
  uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  Ctx c;
  c.sbase = smem_u32(sm);
  c.rank = cluster_rank();
  c.pair = (int)(blockIdx.x >> 1);
  c.n_pairs = (int)(gridDim.x >> 1);
  if (p.pair_off) {  // the host's assignment (longest units first, to the least-loaded pair)
    c.u0 = p.pair_off[c.pair];
    c.u1 = p.pair_off[c.pair + 1];
    c.ustep = 1;
  } else {
    c.u0 = c.pair;
    c.u1 = p.n_units;
    c.ustep = c.n_pairs;
  }
  c.wc = WaitCtl{p.err, p.wait_ns};
  // a launch queued behind this one that reads nothing this one writes may
  // start on each pair this one leaves
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kSmTmemSlot);
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(B_KFULL + b), 4);  // the even CTA's four region lanes (expect_tx: bytes of both halves)
      mbar_init(c.bar(B_VFULL + b), 1);  // the even CTA's chunk-0 lane (expect_tx: every chunk of both CTAs)
      mbar_init(c.bar(B_VEMPTY + b), 1);
      mbar_init(c.bar(B_SCFULL + b), 1);
      mbar_init(c.bar(B_SCEMPTY + b), kSoftmaxWarps);  // every softmax warp, after reading the scales
      mbar_init(c.bar(B_SFULL + b), 1);
      mbar_init(c.bar(B_PFULL + b), 2 * kSoftmaxWarps);
      mbar_init(c.bar(B_STATS + b), kSoftmaxWarps);
    }
    mbar_init(c.bar(B_QFULL), c.rank == 0 ? 5 : 4);  // one arrival per Q region (+ the odd CTA's)
    mbar_init(c.bar(B_QREADY), 4);
    mbar_init(c.bar(B_QREADY2), 8);
    mbar_init(c.bar(B_QEMPTY), 1);
    mbar_init(c.bar(B_OFULL), 1);
    mbar_init(c.bar(B_OEMPTY), 8);
    mbar_init(c.bar(B_STALL), 1);
    mbar_init(c.bar(B_DRAIN), 1);
    mbar_init(c.bar(B_QSOON), 1);
    fence_mbar_init();
    tma_prefetch_map(&m.k);
    tma_prefetch_map(&m.v);
    tma_prefetch_map(&m.q);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  // scale slots start at zero: columns past a tile's width then hold finite
  // stale scales, which the softmax multiplies by p = 0
  for (int i = threadIdx.x; i < 2 * 256; i += kThreads) reinterpret_cast<float*>(sm + kSmScale)[i] = 0.f;
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before either may arrive on the other's
  tc_fence_after();
  c.tb = *tmem_slot;

  const int lane = threadIdx.x & 31;
  if (warp < 4) {
    if (warp == 0) {
      if (lane < kKSlots) role_producer_k(p, m, c, lane);
    } else if (warp == 1) {
      if (lane == 0 && c.rank == 0) role_mma(p, c);
    } else if (warp == 2) {
      if (lane < kVSlots) role_producer_v(p, m, c, lane);
    } else {
      if (lane < 5) role_producer_q(p, m, c, lane);
    }
  } else if (warp < 4 + kSoftmaxWarps) {
    role_softmax(p, c, sm);
  } else {
    role_correction(p, c, sm);
  }
  // the odd CTA's TMEM and shared memory are in use until the pair's last MMA is done
  if (c.rank == 1 && warp == 1 && lane == 0) (void)mbar_wait_drain(c.bar(B_DRAIN), 0, kDrainNs);

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no arrival from the other CTA is still on its way
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(c.tb, 512);
  }
}

// Debug export (tests): the int8 query grid of the fused prologue, run by
// q_codes_int8 itself on rows staged in the layout the Q TMA load writes
// (four 64-dim regions of 128-byte rows, 128-byte swizzle), one thread per row
// as in the correction warps.
constexpr int kDbgQSmem = 4 * kRegionBytes + 1024;

__global__ void __launch_bounds__(kRows) debug_qcodes_kernel(const __nv_bfloat16* q, int n, int8_t* codes,
                                                             float* scales) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  const int r = threadIdx.x;
  const int row = blockIdx.x * kRows + r;
  const uint4* src = reinterpret_cast<const uint4*>(q + (size_t)row * kHeadDim);
#pragma unroll 4
  for (int pc = 0; pc < 32; ++pc) *swz(sm + (pc >> 3) * kRegionBytes, r, pc & 7) = row < n ? src[pc] : make_uint4(0, 0, 0, 0);
  const float s = q_codes_int8(sm, r);
  if (row >= n) return;
  uint32_t* dst = reinterpret_cast<uint32_t*>(codes + (size_t)row * kHeadDim);
#pragma unroll 4
  for (int pc = 0; pc < 32; ++pc) {
    const uint4 v = *swz(sm + (pc >> 3) * kRegionBytes, r, pc & 7);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t b[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {  // two bf16 codes (exact integers) -> two int8 bytes
      const int lo = (int)__uint_as_float(w[e] << 16), hi = (int)__uint_as_float(w[e] & 0xffff0000u);
      b[e] = ((uint32_t)lo & 0xffu) | (((uint32_t)hi & 0xffu) << 8);
    }
    dst[2 * pc] = b[0] | (b[1] << 16);
    dst[2 * pc + 1] = b[2] | (b[3] << 16);
  }
  scales[row] = s;
}

}  // namespace

cudaError_t launch_debug_qcodes(const __nv_bfloat16* q, int n, int8_t* codes, float* scales, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(debug_qcodes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDbgQSmem);
  if (e != cudaSuccess) return e;
  debug_qcodes_kernel<<<(n + kRows - 1) / kRows, kRows, kDbgQSmem, st>>>(q, n, codes, scales);
  return cudaGetLastError();
}

int attention_pairs(int n_sm) {
  static int max_pairs = -1;
  if (max_pairs < 0) {
    if (cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      return imax(1, n_sm / 2);
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * (unsigned)imax(1, n_sm / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kAttnSmem;
    int mc = 0;
    if (cudaOccupancyMaxActiveClusters(&mc, attention_kernel, &cfg) != cudaSuccess || mc <= 0) {
      (void)cudaGetLastError();
      mc = imax(1, n_sm / 2);
    }
    max_pairs = mc;
  }
  return max_pairs;
}

cudaError_t launch_attention(const AttnParams& p, const AttnMaps& m, int n_sm, cudaStream_t st, bool overlap_prev) {
  cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
  if (e != cudaSuccess) return e;
  // persistent grid: one CTA pair per co-resident cluster slot (or per unit),
  // or the pairs the host assigned the units to
  const int pairs = p.pair_off ? p.plan_pairs : imax(1, imin(p.n_units, attention_pairs(n_sm)));
  if (!overlap_prev) {
    attention_kernel<<<2 * pairs, kThreads, kAttnSmem, st>>>(p, m);
    return cudaGetLastError();
  }
  // programmatic dependent launch: its pairs start as the previous attention
  // launch's pairs leave (the two share no data)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * (unsigned)pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attention_kernel, p, m);
}

}  // namespace pa
