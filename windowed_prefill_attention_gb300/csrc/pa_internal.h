// Declarations shared by the C-ABI host code (pa_api.cu) and the kernels
// (pa_kernels.cu).  Not part of the public interface.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "pa_tiles.cuh"

namespace pa {

// One work unit: 256 query rows of one kv head (see pa_tiles.cuh).
struct Unit {
  int seq;      // sequence index
  int g;        // kv head
  int t0;       // absolute first token of the unit (multiple of UT = 256 / G)
  int n_tiles;  // key tiles it visits (its cost)
};

// Inputs of the widening (gather) pass: the paged int8 pool read through the
// block table into contiguous per-kv-head buffers in logical key order.
struct WidenParams {
  const int8_t* k_pool;       // [n_pool][16][HKV][256]
  const int8_t* v_pool;
  const float* k_scale;       // [n_pool][16][HKV]
  const float* v_scale;
  const int32_t* block_table; // [n_seq][bt_stride]
  int bt_stride;
  int n_pool;
  int HKV;
  const SeqGeom* seqs;        // device
  int n_seq;
  int n_stored_blocks;        // sum over sequences of SeqGeom::n_blocks
  int n_tok_cap;              // row stride of the widened buffers
  __nv_bfloat16* kw;          // [HKV][n_tok_cap][256]   integer-valued bf16 K codes
  __half* vt;                 // [HKV][256][n_tok_cap]   integer-valued fp16 V codes, transposed
  float* ks;                  // [HKV][n_tok_cap]        per-token K scale
  float* vs;                  // [HKV][n_tok_cap]        per-token V scale
  unsigned int* vsmax;        // [n_seq][HKV] float bits: max V scale (atomicMax)
  int* err;
  float k_mult = 1.f;         // ks = k_scale * k_mult (the attention folds sm_scale * log2(e) in here)
};

struct AttnParams {
  const __nv_bfloat16* q;     // [total_q][HQ][256]
  int total_q;
  const SeqGeom* seqs;
  const Unit* units;
  int n_units;
  // units assigned to SM pairs by the host: pair i runs units [pair_off[i],
  // pair_off[i + 1]) on a grid of plan_pairs pairs; plan_pairs = 0: pair i runs
  // units i, i + n_pairs, ... of the list
  const int* pair_off;
  int plan_pairs;
  const float* ks;
  const float* vs;
  const unsigned int* vsmax;
  __nv_bfloat16* out;         // [total_q][HQ][256]
  const __nv_bfloat16* gate;  // [total_q][HQ][256] output gate (sigmoid), or nullptr
  int HQ, HKV, G, TQ;         // TQ = 128 / G: tokens per CTA, half a unit
  int n_tok_cap;
  int S, W;
  float sm_scale_log2;        // sm_scale * log2(e), already folded into ks
  int q_mode, p_mode;
  int* err;
  unsigned long long wait_ns;
  const unsigned int* q_ready;  // nullptr, or a word that equals q_epoch once q holds the units' rows
  unsigned int q_epoch;
  int debug_stall;            // test hook: first wait targets a barrier nothing arrives at
};

struct AttnMaps {
  CUtensorMap k;   // Kw  [HKV][n_tok][256] bf16, box {64, 64, 1}: one CTA's keys of a 64-dim region of a key tile
  CUtensorMap v;   // Vt  [HKV][256][n_tok] fp16, box {64, 128, 1}: one CTA's dims of a 64-key chunk
  CUtensorMap q;   // q   [tokens][HQ][256] bf16, box {64, G, TQ}: one region of a CTA's 128 rows
};

// Launchers (return the launch's cudaError_t).
cudaError_t launch_widen(const WidenParams& p, cudaStream_t st);

// KV append: the new tokens' K/V rows quantised into the pool.
struct KvAppendParams {
  const __nv_bfloat16* k_new;  // [n_new][HKV][256]
  const __nv_bfloat16* v_new;  // [n_new][HKV][256]
  int n_new, tok_start, HKV, n_pool;
  const int32_t* bt_row;       // pool page of each 16-token block of the sequence
  int8_t* k_pool;
  int8_t* v_pool;
  float* k_scale;
  float* v_scale;
  int* err;
};
cudaError_t launch_kv_append(const KvAppendParams& p, cudaStream_t st);

// Decode: one query token per sequence.  The launch's (sequence, kv head)
// pairs laid end to end give a list of visible 16-token blocks; each CTA takes
// a run of it, which may cover the end of one pair and the start of the next:
// runs of equal cost listed in the launch's parameters (one-wave grids), else
// equal runs of per_cta blocks.
constexpr int kDecMaxCtaBlocks = 128;  // blocks per CTA at most: 32 per warp
constexpr int kDecPartStride = 260;    // floats per partial row: max (log2), sum, 2 pad, O[256]
constexpr int kDecParamSeqs = 512;     // sequences per launch, their table carried in the launch's parameters
// One launch's sequences, passed by value (no upload per call):
// {row of the token in q / out, context length, visible blocks of the launch's
// earlier sequences (per kv head), 0}; the token is the context's last.
constexpr int kDecParamCtas = 512;    // CTA runs the launch's parameters can carry
struct DecodeSeqs {
  int4 seq[kDecParamSeqs];
  int cta_x0[kDecParamCtas];          // first block of CTA c's run (the run ends where CTA c + 1's starts)
  uint16_t cta_seq[kDecParamCtas];    // sequence of that block
  uint16_t cta_slot[kDecParamCtas];   // CTA c's partial slot in that block's pair (CTAs before it in the pair)
};
struct DecodeParams {
  const __nv_bfloat16* q;  // [rows][HQ][256]
  __nv_bfloat16* out;      // [rows][HQ][256]
  const int8_t* k_pool;
  const int8_t* v_pool;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  int bt_stride, n_pool;
  int n_seq;               // sequences of this launch (<= kDecParamSeqs)
  int bt_row0;             // block-table row of the launch's first sequence
  int S, W;                // sink blocks, window blocks (W <= 0: no window)
  int HQ, HKV, G;
  int total;               // visible blocks of all pairs of the launch
  int per_cta;             // blocks per CTA (<= kDecMaxCtaBlocks) when runs_listed is 0
  int max_slots;           // partial slots per pair
  int runs_listed;         // DecodeSeqs::cta_* hold every CTA's run
  float sm_scale_log2;
  float* part;             // [n_seq * HKV][max_slots][G][kDecPartStride]
  // [n_seq * HKV] per pair: low 32 bits the blocks of the partials written so
  // far, high 32 bits its partial count (added by the CTA that holds its last
  // block); 0 between launches (the merging CTA resets it)
  unsigned long long* tickets;
  int* err;
  unsigned long long wait_ns;  // bound on every wait for a copy
};
// The pool as the decode kernel's TMA copies see it: uint8 [n_pool * 16][HKV][256],
// box {128, 1, 16} (one kv head's 16 tokens of a page, half the dims), 128-byte swizzle.
struct DecodeMaps {
  CUtensorMap k;
  CUtensorMap v;
};
cudaError_t launch_decode(const DecodeParams& p, const DecodeSeqs& seqs, const DecodeMaps& m, int n_cta,
                          cudaStream_t st);
// Decode CTAs that fit on one SM at a time for HKV kv heads (occupancy, cached).
int decode_ctas_per_sm(int HKV);
// overlap_prev: the launch may start while the previous attention launch on
// `st` is still running (it must read nothing that launch writes).
cudaError_t launch_attention(const AttnParams& p, const AttnMaps& m, int n_sm, cudaStream_t st,
                             bool overlap_prev = false);
// CTA pairs of the attention kernel that run at once (its persistent grid).
int attention_pairs(int n_sm);

// Debug exports (tests only).
cudaError_t launch_debug_gather(const WidenParams& p, int seq, int8_t* k_out, int8_t* v_out, float* ks_out,
                                float* vs_out, int32_t* tok_out, cudaStream_t st);
// The int8 query grid of the attention prologue on n rows of 256 bf16 values:
// codes int8 [n][256], scales fp32 [n].
cudaError_t launch_debug_qcodes(const __nv_bfloat16* q, int n, int8_t* codes, float* scales, cudaStream_t st);
cudaError_t launch_debug_maskset(const SeqGeom* seqs, const Unit* units, int n_units, int UT, int G, int S, int W,
                                 int32_t* row_counts, int32_t* unit_blocks, int cap, cudaStream_t st);

}  // namespace pa
