// Work-unit and key-tile geometry of the windowed prefill attention, shared
// by the host planner and every kernel (one definition, so the planner's tile
// counts, the producer's loads, the MMA issuer and the softmax agree).
//
// Mask ("int8 tensor-core prefill attention", section "Why the attention, and
// why tensor cores"; "Relation to open PRs" for the window-off case): query
// token t sees key j iff j <= t and, when the window is on (W > 0), j's 16-token
// block is a sink block (< S) or lies in the last W blocks up to t's own block,
// i.e. block(j) >= max(0, block(t) + 1 - W).  The window start is a function of
// block(t) only, so it is constant over a 16-row query tile and only the
// causal bound varies per row.
//
// A work unit is 256 query rows of one kv head g, one 256-row MMA over a pair
// of CTAs: UT = 256 / G consecutive tokens times the G q heads that share g
// (row r = token_in_unit * G + head_in_group); each CTA holds 128 rows, the
// first or second TQ = UT / 2 tokens.  Units start on absolute multiples of UT,
// so for G = 8 a unit is two 16-token query blocks (the pages' 16-row tiles).
// Both halves of a unit visit the same key tiles: those of the union of the
// unit's query blocks; the per-row mask hides what a row may not see.
//
// Key tiles: the unit's visible key blocks form at most two runs, the sink run
// [0, S) and the window run [lo(first block), last block]; when they touch they
// merge into one run from block 0.  Each run is cut into tiles of up to
// kTileBlocks 16-key blocks (128 keys).  Masked blocks are never visited.
#pragma once

#ifdef __CUDACC__
#define PA_HD __host__ __device__ __forceinline__
#else
#define PA_HD inline
#endif

namespace pa {

constexpr int kPage = 16;         // tokens per KV page (= mask block)
constexpr int kHeadDim = 256;     // head dimension
constexpr int kRows = 128;        // query rows per CTA (TMEM lanes)
constexpr int kUnitRows = 2 * kRows;  // query rows per work unit (MMA M over a CTA pair)
constexpr int kTileBlocks = 8;    // 16-key blocks per key tile
constexpr int kTileKeys = kTileBlocks * kPage;  // 128
constexpr int kChunkKeys = 64;    // keys per V^T chunk (PV works through a tile in chunks)

PA_HD int imin(int a, int b) { return a < b ? a : b; }
PA_HD int imax(int a, int b) { return a > b ? a : b; }

// Per-sequence description, host-computed, read by the kernels.
struct SeqGeom {
  int q_off;       // first row of the sequence in q / out
  int q_start;     // absolute position of that row
  int n_q;         // query tokens
  int n_ctx;       // context tokens (q_start + n_q)
  int tok_off;     // first row of the sequence in the widened K/V buffers
  int vis_lo;      // first window block any query of the call can see (0 if W <= 0)
  int n_sink_vis;  // sink blocks stored ahead of vis_lo: min(S, vis_lo) (0 if W <= 0)
  int n_blocks;    // blocks stored in the widened buffers for this sequence
  int bt_row;      // row of this sequence in the block table
  int pad[3];
};

// Widened-buffer geometry of one sequence.  Blocks below vis_lo that are not
// sink blocks can never be seen by any query of this call and are not stored.
PA_HD void seq_geom_fill(SeqGeom& s, int S, int W) {
  const int last_blk = (s.q_start + s.n_q - 1) / kPage;
  if (W > 0) {
    s.vis_lo = imax(0, s.q_start / kPage + 1 - W);
    s.n_sink_vis = imin(S, s.vis_lo);
  } else {
    s.vis_lo = 0;
    s.n_sink_vis = 0;
  }
  s.n_blocks = s.n_sink_vis + (last_blk - s.vis_lo + 1);
}

// Stored block index (within the sequence) -> logical key block.
PA_HD int stored_to_logical_block(const SeqGeom& s, int b) {
  return b < s.n_sink_vis ? b : s.vis_lo + (b - s.n_sink_vis);
}
// Logical key block -> first widened row (global, all sequences).
PA_HD int logical_block_row(const SeqGeom& s, int kb) {
  const int b = kb < s.vis_lo ? kb : s.n_sink_vis + (kb - s.vis_lo);
  return s.tok_off + b * kPage;
}

// Geometry of one work unit.
struct UnitGeom {
  int ta, tb;          // first / last query token of the unit inside the sequence's query range
  int qa, qb;          // their 16-token blocks
  int lo_b;            // window start of the last block (0 if W <= 0)
  int nsk;             // blocks of the separate sink run (0 if merged or no window)
  int ws;              // first block of the window run
  int n_sink_tiles;    // tiles of the sink run
  int n_tiles;         // all tiles
};

PA_HD UnitGeom unit_geom(int t0, int TQ, const SeqGeom& s, int S, int W) {
  UnitGeom u;
  u.ta = imax(t0, s.q_start);
  u.tb = imin(t0 + TQ, s.q_start + s.n_q) - 1;
  u.qa = u.ta / kPage;
  u.qb = u.tb / kPage;
  int lo_a = 0;
  u.lo_b = 0;
  if (W > 0) {
    lo_a = imax(0, u.qa + 1 - W);
    u.lo_b = imax(0, u.qb + 1 - W);
  }
  const bool separate = W > 0 && lo_a > S;
  u.nsk = separate ? S : 0;
  u.ws = separate ? lo_a : 0;
  u.n_sink_tiles = (u.nsk + kTileBlocks - 1) / kTileBlocks;
  u.n_tiles = u.n_sink_tiles + (u.qb + 1 - u.ws + kTileBlocks - 1) / kTileBlocks;
  return u;
}

struct TileGeom {
  int kb0;         // first logical key block
  int nb;          // blocks in the tile (1..kTileBlocks)
  bool needs_mask; // some row of the unit does not see some key of the tile
};

PA_HD TileGeom tile_geom(const UnitGeom& u, int i, int S, int W) {
  TileGeom g;
  if (i < u.n_sink_tiles) {
    g.kb0 = i * kTileBlocks;
    g.nb = imin(kTileBlocks, u.nsk - g.kb0);
  } else {
    g.kb0 = u.ws + (i - u.n_sink_tiles) * kTileBlocks;
    g.nb = imin(kTileBlocks, u.qb + 1 - g.kb0);
  }
  const int kb1 = g.kb0 + g.nb;  // exclusive
  // causal: blocks at or after the unit's first query block are partly hidden
  // from its earlier rows; window: non-sink blocks below the last block's
  // window start are hidden from the later rows.
  g.needs_mask = (kb1 - 1 >= u.qa) || (W > 0 && imax(g.kb0, S) < imin(kb1, u.lo_b));
  return g;
}

// Width in blocks of tile i, the same as tile_geom(u, i, S, W).nb: only the
// last tile of each run can be narrower than kTileBlocks.  Written as selects
// (no branch): the MMA issuer evaluates it per tile on its critical path.
PA_HD int tile_width(const UnitGeom& u, int i) {
  int w = kTileBlocks;
  w = i == u.n_sink_tiles - 1 ? u.nsk - i * kTileBlocks : w;
  w = i == u.n_tiles - 1 ? (u.qb + 1 - u.ws) - (u.n_tiles - 1 - u.n_sink_tiles) * kTileBlocks : w;
  return w;
}

// Bits [0, n) set, for n clamped to [0, 64].
PA_HD unsigned long long low_bits(int n) {
  return n <= 0 ? 0ull : (n >= 64 ? ~0ull : ((1ull << n) - 1ull));
}

// Which of the 64 key columns [64 half, 64 half + 64) of a tile query token t
// sees, as a bit mask: the tile's width and, where the tile needs masking, the
// causal bound (key <= t) and the sink / window test (key block < S, or
// >= lo = max(0, t/16 + 1 - W)).  This is the mask the softmax applies, one
// bit test per score.
PA_HD unsigned long long visible_columns(const TileGeom& tg, int t, int S, int W, int half) {
  const int key0 = tg.kb0 * kPage + 64 * half;
  unsigned long long v = low_bits(tg.nb * kPage - 64 * half);
  if (tg.needs_mask) {
    v &= low_bits(t - key0 + 1);
    if (W > 0) {
      const int lo = imax(0, t / kPage + 1 - W);
      v &= low_bits(S * kPage - key0) | ~low_bits(lo * kPage - key0);
    }
  }
  return v;
}

}  // namespace pa
