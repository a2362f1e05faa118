// C-ABI host side: handle, argument checks, the window-aware work planner
// (longest-first unit order), workspace, tensor maps and launches.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

using namespace pa;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

typedef CUresult (*WriteValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

// cuStreamWriteValue32: a 32-bit store that a stream performs in order with
// its copies (after a memory barrier), without a kernel
WriteValue32Fn write_value_fn() {
  static WriteValue32Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WriteValue32Fn>(p);
  });
  return fn;
}

struct Plan {
  std::vector<SeqGeom> seqs;
  std::vector<Unit> units;
  std::vector<int> pair_off;  // when the units are assigned to pairs: pair i's first unit (assign_pairs)
  int n_pairs = 0;
  int n_stored_blocks = 0;
  int n_tok_total = 0;
  int total_q = 0;
  long long n_tiles = 0;
};

// Host planner: per-sequence widened geometry and the work units sorted by
// decreasing cost (tiles), so the longest units start first.
int build_plan(int HQ, int HKV, int n_seq, const pa_seq* seqs, int S, int W, int max_pages, Plan& P) {
  if (HQ <= 0 || HKV <= 0 || HQ % HKV != 0) return PA_EINVAL;
  const int G = HQ / HKV;
  if (G > kRows || kRows % G != 0) return PA_EINVAL;
  if (n_seq <= 0 || seqs == nullptr || S < 0) return PA_EINVAL;
  const int UT = kUnitRows / G;  // tokens per unit
  P = Plan();
  int tok_off = 0;
  for (int s = 0; s < n_seq; ++s) {
    const pa_seq& q = seqs[s];
    if (q.n_q < 1 || q.q_start < 0 || q.q_off < 0 || q.n_ctx < q.q_start + q.n_q) return PA_EINVAL;
    if (max_pages > 0 && (long long)q.n_ctx > (long long)max_pages * kPage) return PA_EINVAL;
    if ((long long)q.q_off + q.n_q > (1LL << 30) || (long long)q.n_ctx > (1LL << 30)) return PA_EINVAL;
    SeqGeom g{};
    g.q_off = q.q_off;
    g.q_start = q.q_start;
    g.n_q = q.n_q;
    g.n_ctx = q.n_ctx;
    g.tok_off = tok_off;
    g.bt_row = s;
    seq_geom_fill(g, S, W);
    tok_off += g.n_blocks * kPage;
    if (tok_off > (1 << 30)) return PA_EINVAL;
    P.seqs.push_back(g);
    P.total_q = std::max(P.total_q, q.q_off + q.n_q);
    const int t_first = (q.q_start / UT) * UT;
    for (int t0 = t_first; t0 < q.q_start + q.n_q; t0 += UT) {
      const UnitGeom ug = unit_geom(t0, UT, g, S, W);
      for (int kv = 0; kv < HKV; ++kv) {
        P.units.push_back(Unit{s, kv, t0, ug.n_tiles});
        P.n_tiles += ug.n_tiles;
      }
    }
  }
  std::stable_sort(P.units.begin(), P.units.end(), [](const Unit& a, const Unit& b) { return a.n_tiles > b.n_tiles; });
  P.n_stored_blocks = tok_off / kPage;
  P.n_tok_total = tok_off;
  return PA_OK;
}

// A pair's change of unit costs about two tiles' time (the unit's last PV and
// the epilogue, the next unit's Q rows and first QK^T; clock64 stamps on
// GB300), so a unit weighs its tiles plus that.
constexpr int kUnitSwitchTiles = 2;
// The attention kernel's pairs for n units: one per co-resident cluster slot,
// at most one per unit.
int launch_pairs(int n_sm, int n) { return std::max(1, std::min(n, pa::attention_pairs(n_sm))); }
// Unit records (16 bytes) that hold n_pairs + 1 pair offsets after a unit list.
size_t pair_off_records(int n_pairs) { return ((size_t)n_pairs + 1 + 3) / 4; }
// Units sorted longest first, assigned to n_pairs SM pairs: each to the pair
// whose work so far is least (ties: the lowest pair), a greedy
// longest-first schedule; then laid out pair by pair, each pair's units still
// longest first.  off[i] = pair i's first unit, off[n_pairs] = n.  Against
// walking the sorted list with stride n_pairs (pair i: units i, i + n_pairs,
// ...), the most loaded pair's work falls from 1.28x the mean to 1.04x at 4k
// tokens (256 units), 1.09x to 1.01x for the chunked batch, 1.02x to 1.00x at
// 32k.
void assign_pairs(const Unit* units, int n, int n_pairs, std::vector<Unit>& out, std::vector<int>& off) {
  using Load = std::pair<long long, int>;  // (work so far, pair)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> q;
  for (int i = 0; i < n_pairs; ++i) q.push(Load{0, i});
  std::vector<int> pair_of((size_t)n);
  std::vector<int> count((size_t)n_pairs, 0);
  for (int u = 0; u < n; ++u) {
    const Load top = q.top();
    q.pop();
    pair_of[(size_t)u] = top.second;
    ++count[(size_t)top.second];
    q.push(Load{top.first + units[u].n_tiles + kUnitSwitchTiles, top.second});
  }
  off.assign((size_t)n_pairs + 1, 0);
  for (int i = 0; i < n_pairs; ++i) off[(size_t)i + 1] = off[(size_t)i] + count[(size_t)i];
  out.resize((size_t)n);
  std::vector<int> next(off.begin(), off.end() - 1);
  for (int u = 0; u < n; ++u) out[(size_t)next[(size_t)pair_of[(size_t)u]]++] = units[u];
}

bool same_plan_key(const std::vector<int>& a, const std::vector<int>& b) { return a == b; }

// The host-buffer path's chunks: ends (rows of the sequences laid end to end)
// of chunks of work units counted in waves (a wave: one unit for every one of
// the n_pairs SM pairs the kernel runs at once; a part-filled wave leaves
// pairs idle): one wave first and one wave last, two in between.  The short
// first chunk starts the computation and the copy-out early, the short last
// one shortens what is left after the last rows are in; two waves between
// keep the launches few (at 32k tokens on GB300: 921 TOPS end to end against
// 888 with two-wave chunks throughout, 896-904 with three-wave middles or
// half-wave ends).  A boundary inside a sequence moves to a multiple of a
// unit's tokens (down, or up to the sequence's end when that would empty the
// piece), so every unit lies in one chunk.  ends is increasing, last = total rows.
int host_chunk_ends(int HQ, int HKV, int n_seq, const pa_seq* seqs, int n_pairs, std::vector<long long>& ends) {
  if (HQ <= 0 || HKV <= 0 || HQ % HKV != 0 || kUnitRows % (HQ / HKV) != 0) return PA_EINVAL;
  if (n_seq <= 0 || seqs == nullptr || n_pairs <= 0) return PA_EINVAL;
  std::vector<long long> base(n_seq + 1, 0);  // first row of each sequence, end to end
  for (int s = 0; s < n_seq; ++s) {
    if (seqs[s].n_q < 1 || seqs[s].q_start < 0) return PA_EINVAL;
    base[s + 1] = base[s] + seqs[s].n_q;
  }
  const long long T = base[n_seq];
  const long long UT = kUnitRows / (HQ / HKV);  // tokens per unit
  const long long wave = std::max(UT, (long long)n_pairs * UT / HKV);
  std::vector<long long> cuts;
  for (long long at = 0; at < T;) {
    long long step = at == 0 ? wave : 2 * wave;
    if (T - at > wave && T - at - step < wave) step = T - at - wave;  // a last chunk of one wave
    at = std::min(T, at + step);
    cuts.push_back(at);
  }
  ends.clear();
  for (long long cut : cuts) {
    const int s = (int)(std::upper_bound(base.begin(), base.end(), cut) - base.begin()) - 1;
    if (s >= 0 && s < n_seq && cut != base[s]) {  // inside sequence s
      const long long abs_pos = seqs[s].q_start + (cut - base[s]);
      long long r = abs_pos / UT * UT;
      if (r <= seqs[s].q_start) r = std::min((long long)seqs[s].q_start + seqs[s].n_q, (abs_pos / UT + 1) * UT);
      cut = base[s] + (r - seqs[s].q_start);
    }
    if (ends.empty() || cut > ends.back()) ends.push_back(cut);
  }
  return PA_OK;
}

}  // namespace

struct pa_ctx {
  int HQ = 0, HKV = 0, G = 0, TQ = 0, n_pool = 0, max_pages = 0;
  pa_options opt{};
  int device = 0, n_sm = 0;

  // workspace
  __nv_bfloat16* kw = nullptr;
  __half* vt = nullptr;
  float* ks = nullptr;
  float* vs = nullptr;
  int n_tok_cap = 0;
  unsigned int* vsmax = nullptr;
  int vsmax_cap = 0;
  SeqGeom* d_seqs = nullptr;
  int seqs_cap = 0;
  Unit* d_units = nullptr;
  int units_cap = 0;
  int* d_err = nullptr;
  unsigned int* d_qflags = nullptr;  // host path: chunk c's q rows are in when d_qflags[c] == q_epoch
  int qflags_cap = 0;
  unsigned int q_epoch = 0;

  // plan upload through pinned staging
  void* h_stage = nullptr;
  size_t h_stage_cap = 0;
  cudaEvent_t upload_done = nullptr;
  bool upload_recorded = false;
  std::vector<int> plan_key;
  Plan plan;

  // tensor maps
  AttnMaps maps{};
  const void* kv_ptr = nullptr;
  int kv_rows = -1;
  int kv_cap = -1;

  // decode: partials, the pairs' tickets (zeroed once; the kernel leaves them
  // at zero), the pool's tensor maps (cached by pool pointers)
  DecodeMaps dec_maps{};
  const void* dec_kp = nullptr;
  const void* dec_vp = nullptr;
  float* d_part = nullptr;
  int part_cap = 0;
  unsigned long long* d_tickets = nullptr;
  int tickets_cap = 0;

  // host-buffer path staging
  void* hb[7] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  size_t hb_cap[7] = {0, 0, 0, 0, 0, 0, 0};
  cudaStream_t s_h2d = nullptr, s_d2h = nullptr;  // the host path's copy streams
  std::vector<cudaEvent_t> pipe_ev;                // and its events (no timing)
  SeqGeom* d_pseqs = nullptr;                      // its chunks' plans, uploaded together
  int pseqs_cap = 0;
  Unit* d_punits = nullptr;
  int punits_cap = 0;
  void* h_pstage = nullptr;
  size_t h_pstage_cap = 0;
  cudaEvent_t pstage_done = nullptr;
  bool pstage_recorded = false;

  // timing
  std::vector<cudaEvent_t> ev_free;
  std::vector<cudaEvent_t> ev_pending;  // triples (before widen, after widen, after attention)
  double t_widen = 0.0, t_attn = 0.0;
  int t_calls = 0;
};

namespace {

int cuda_fail(cudaError_t e) {
  if (e == cudaErrorMemoryAllocation) return PA_ENOMEM;
  return PA_ECUDA;
}

#define PA_CUDA(x)                              \
  do {                                          \
    cudaError_t e_ = (x);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)

template <typename T>
int grow(T*& p, int& cap, size_t need) {
  if ((size_t)cap >= need) return PA_OK;
  size_t n = std::max(need, (size_t)cap + (size_t)cap / 2);
  if (p) PA_CUDA(cudaFree(p));
  p = nullptr;
  cap = 0;
  PA_CUDA(cudaMalloc(reinterpret_cast<void**>(&p), n * sizeof(T)));
  cap = (int)n;
  return PA_OK;
}

int grow_bytes(void*& p, size_t& cap, size_t need) {
  if (cap >= need) return PA_OK;
  size_t n = std::max(need, cap + cap / 2);
  if (p) PA_CUDA(cudaFree(p));
  p = nullptr;
  cap = 0;
  PA_CUDA(cudaMalloc(&p, n));
  cap = n;
  return PA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A decode launch's CTA runs: first block, its sequence, the CTA's partial slot in its pair.
struct DecRuns {
  std::vector<int> x0, seq, slot;
  int max_slots = 1;
};

int encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
           const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ECUDA;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ECUDA;
}

// Plan (cached by its inputs), workspace sizing and the upload of the plan.
// Widened-row workspace for at least `rows` rows (reallocating frees the old
// buffers, which waits for the device).
int reserve_rows(pa_handle h, size_t rows) {
  const size_t need_tok = (rows + 63) / 64 * 64;
  if ((size_t)h->n_tok_cap >= need_tok) return PA_OK;
  size_t cap = std::max(need_tok, (size_t)h->n_tok_cap + (size_t)h->n_tok_cap / 2);
  cap = (cap + 63) / 64 * 64;
  if (h->kw) cudaFree(h->kw);
  if (h->vt) cudaFree(h->vt);
  if (h->ks) cudaFree(h->ks);
  if (h->vs) cudaFree(h->vs);
  h->kw = nullptr;
  h->vt = nullptr;
  h->ks = nullptr;
  h->vs = nullptr;
  h->n_tok_cap = 0;
  h->kv_ptr = nullptr;
  PA_CUDA(cudaMalloc(&h->kw, cap * h->HKV * kHeadDim * sizeof(__nv_bfloat16)));
  PA_CUDA(cudaMalloc(&h->vt, cap * h->HKV * kHeadDim * sizeof(__half)));
  PA_CUDA(cudaMalloc(&h->ks, cap * h->HKV * sizeof(float)));
  PA_CUDA(cudaMalloc(&h->vs, cap * h->HKV * sizeof(float)));
  h->n_tok_cap = (int)cap;
  return PA_OK;
}

int prepare(pa_handle h, int n_seq, const pa_seq* seqs, int S, int W, cudaStream_t st) {
  std::vector<int> key;
  key.reserve(4 + 4 * n_seq);
  key.push_back(n_seq);
  key.push_back(S);
  key.push_back(W);
  for (int s = 0; s < n_seq; ++s) {
    key.push_back(seqs[s].q_off);
    key.push_back(seqs[s].q_start);
    key.push_back(seqs[s].n_q);
    key.push_back(seqs[s].n_ctx);
  }
  if (!h->plan_key.empty() && same_plan_key(key, h->plan_key)) return PA_OK;
  Plan P;
  int rc = build_plan(h->HQ, h->HKV, n_seq, seqs, S, W, h->max_pages, P);
  if (rc) return rc;
  // the units laid out pair by pair for the kernel's pairs, the pair offsets after them
  const int n_u = (int)P.units.size();
  P.n_pairs = launch_pairs(h->n_sm, n_u);
  {
    std::vector<Unit> by_pair;
    assign_pairs(P.units.data(), n_u, P.n_pairs, by_pair, P.pair_off);
    P.units = std::move(by_pair);
  }
  const size_t n_rec = (size_t)n_u + pair_off_records(P.n_pairs);
  // workspace
  if ((rc = reserve_rows(h, (size_t)P.n_tok_total))) return rc;
  if ((rc = grow(h->vsmax, h->vsmax_cap, (size_t)n_seq * h->HKV))) return rc;
  if ((rc = grow(h->d_seqs, h->seqs_cap, P.seqs.size()))) return rc;
  if ((rc = grow(h->d_units, h->units_cap, n_rec))) return rc;
  // upload through pinned staging; never overwrite staging a copy may still read
  const size_t bytes_s = P.seqs.size() * sizeof(SeqGeom), bytes_u = n_rec * sizeof(Unit);
  if (h->upload_recorded) PA_CUDA(cudaEventSynchronize(h->upload_done));
  if (h->h_stage_cap < bytes_s + bytes_u) {
    if (h->h_stage) cudaFreeHost(h->h_stage);
    h->h_stage = nullptr;
    h->h_stage_cap = 0;
    PA_CUDA(cudaMallocHost(&h->h_stage, bytes_s + bytes_u));
    h->h_stage_cap = bytes_s + bytes_u;
  }
  std::memcpy(h->h_stage, P.seqs.data(), bytes_s);
  std::memcpy(static_cast<char*>(h->h_stage) + bytes_s, P.units.data(), (size_t)n_u * sizeof(Unit));
  std::memcpy(static_cast<char*>(h->h_stage) + bytes_s + (size_t)n_u * sizeof(Unit), P.pair_off.data(),
              P.pair_off.size() * sizeof(int));
  PA_CUDA(cudaMemcpyAsync(h->d_seqs, h->h_stage, bytes_s, cudaMemcpyHostToDevice, st));
  PA_CUDA(cudaMemcpyAsync(h->d_units, static_cast<char*>(h->h_stage) + bytes_s, bytes_u, cudaMemcpyHostToDevice, st));
  PA_CUDA(cudaEventRecord(h->upload_done, st));
  h->upload_recorded = true;
  h->plan = std::move(P);
  h->plan_key = std::move(key);
  return PA_OK;
}

int check_inputs(pa_handle h, const void* q, const int8_t* kp, const int8_t* vp, const float* ksc, const float* vsc,
                 const int32_t* bt, const void* out) {
  if (!h) return PA_EINVAL;
  if (!q || !kp || !vp || !ksc || !vsc || !bt || !out) return PA_EINVAL;
  if (!aligned(q, 16) || !aligned(kp, 16) || !aligned(vp, 16) || !aligned(out, 16)) return PA_EINVAL;
  if (!aligned(ksc, 4) || !aligned(vsc, 4) || !aligned(bt, 4)) return PA_EINVAL;
  return PA_OK;
}

WidenParams widen_params(pa_handle h, const int8_t* kp, const int8_t* vp, const float* ksc, const float* vsc,
                         const int32_t* bt, int n_seq, const SeqGeom* d_seqs = nullptr, int n_stored_blocks = -1) {
  WidenParams w{};
  w.k_pool = kp;
  w.v_pool = vp;
  w.k_scale = ksc;
  w.v_scale = vsc;
  w.block_table = bt;
  w.bt_stride = h->max_pages;
  w.n_pool = h->n_pool;
  w.HKV = h->HKV;
  w.seqs = d_seqs ? d_seqs : h->d_seqs;
  w.n_seq = n_seq;
  w.n_stored_blocks = n_stored_blocks >= 0 ? n_stored_blocks : h->plan.n_stored_blocks;
  w.n_tok_cap = h->n_tok_cap;
  w.kw = h->kw;
  w.vt = h->vt;
  w.ks = h->ks;
  w.vs = h->vs;
  w.vsmax = h->vsmax;
  w.err = h->d_err;
  return w;
}

cudaEvent_t take_event(pa_handle h) {
  if (!h->ev_free.empty()) {
    cudaEvent_t e = h->ev_free.back();
    h->ev_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// The widening pass of plan P, whose sequence table is already on the device
// at d_seqs (the caller has sized the widened workspace for P).
int launch_widen_plan(pa_handle h, const Plan& P, const SeqGeom* d_seqs, int n_seq, const int8_t* kp,
                      const int8_t* vp, const float* ksc, const float* vsc, const int32_t* bt, float sm_scale,
                      cudaStream_t st) {
  PA_CUDA(cudaMemsetAsync(h->vsmax, 0, sizeof(unsigned int) * n_seq * h->HKV, st));
  WidenParams wp = widen_params(h, kp, vp, ksc, vsc, bt, n_seq, d_seqs, P.n_stored_blocks);
  wp.k_mult = sm_scale * 1.4426950408889634f;  // the softmax's sm_scale * log2(e), folded into the K scales
  PA_CUDA(launch_widen(wp, st));
  return PA_OK;
}

// The attention kernel over n_units work units at d_units, all of plan P
// (whose sequence table is on the device at d_seqs and whose pages the
// widening pass has already written).
int launch_attention_plan(pa_handle h, const Plan& P, const SeqGeom* d_seqs, const Unit* d_units, int n_units,
                          const void* q, int S, int W, float sm_scale, void* out, cudaStream_t st,
                          const void* gate, bool overlap_prev = false, const unsigned int* q_ready = nullptr,
                          unsigned int q_epoch = 0, const int* d_pair_off = nullptr, int plan_pairs = 0) {
  int rc = PA_OK;
  // tensor maps
  if (h->kw != h->kv_ptr || P.n_tok_total != h->kv_rows || h->n_tok_cap != h->kv_cap) {
    const uint64_t kd[3] = {(uint64_t)kHeadDim, (uint64_t)P.n_tok_total, (uint64_t)h->HKV};
    const uint64_t kst[2] = {(uint64_t)kHeadDim * 2, (uint64_t)h->n_tok_cap * kHeadDim * 2};
    const uint32_t kbox[3] = {64, (uint32_t)kTileKeys / 2, 1};  // one CTA's half of a tile
    if ((rc = encode(&h->maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, h->kw, kd, kst, kbox,
                     CU_TENSOR_MAP_SWIZZLE_128B)))
      return rc;
    const uint64_t vd[3] = {(uint64_t)P.n_tok_total, (uint64_t)kHeadDim, (uint64_t)h->HKV};
    const uint64_t vst[2] = {(uint64_t)h->n_tok_cap * 2, (uint64_t)h->n_tok_cap * kHeadDim * 2};
    const uint32_t vbox[3] = {(uint32_t)kChunkKeys, (uint32_t)kHeadDim / 2, 1};  // one CTA's half of the dims
    if ((rc = encode(&h->maps.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, h->vt, vd, vst, vbox,
                     CU_TENSOR_MAP_SWIZZLE_128B)))
      return rc;
    h->kv_ptr = h->kw;
    h->kv_rows = P.n_tok_total;
    h->kv_cap = h->n_tok_cap;
  }
  // the query's map: q as [tokens][HQ][256], a unit's rows are TQ tokens x G heads
  AttnMaps maps = h->maps;
  {
    const uint64_t qd[3] = {(uint64_t)kHeadDim, (uint64_t)h->HQ, (uint64_t)P.total_q};
    const uint64_t qst[2] = {(uint64_t)kHeadDim * 2, (uint64_t)h->HQ * kHeadDim * 2};
    const uint32_t qbox[3] = {64, (uint32_t)h->G, (uint32_t)h->TQ};
    if ((rc = encode(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, qd, qst, qbox, CU_TENSOR_MAP_SWIZZLE_128B)))
      return rc;
  }
  AttnParams a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.total_q = P.total_q;
  a.seqs = d_seqs;
  a.units = d_units;
  a.n_units = n_units;
  a.pair_off = d_pair_off;
  a.plan_pairs = plan_pairs;
  a.ks = h->ks;
  a.vs = h->vs;
  a.vsmax = h->vsmax;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.gate = static_cast<const __nv_bfloat16*>(gate);
  a.HQ = h->HQ;
  a.HKV = h->HKV;
  a.G = h->G;
  a.TQ = h->TQ;
  a.n_tok_cap = h->n_tok_cap;
  a.S = S;
  a.W = W;
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  a.q_mode = h->opt.q_mode;
  a.p_mode = h->opt.p_mode;
  a.err = h->d_err;
  a.wait_ns = (unsigned long long)h->opt.wait_timeout_ms * 1000000ull;
  a.q_ready = q_ready;
  a.q_epoch = q_epoch;
  a.debug_stall = h->opt.debug_stall;
  PA_CUDA(launch_attention(a, maps, h->n_sm, st, overlap_prev));
  return PA_OK;
}

// Events for pa_timing around a widening pass and the attention work after
// it: mark(0) before the pass, mark(1) after it, mark(2) after the attention.
struct TimingMarks {
  cudaEvent_t e[3] = {nullptr, nullptr, nullptr};
  bool queued = false;  // mark(2) handed the events to the pending list
  // events of a call that failed before its last mark go back to the free list
  void release(pa_handle h) {
    if (queued) return;
    for (auto& x : e)
      if (x) h->ev_free.push_back(x);
    e[0] = e[1] = e[2] = nullptr;
  }
  int init(pa_handle h) {
    if (!h->opt.record_timing) return PA_OK;
    for (auto& x : e)
      if (!(x = take_event(h))) return PA_ECUDA;
    return PA_OK;
  }
  int mark(pa_handle h, int i, cudaStream_t st) {
    if (!e[i]) return PA_OK;
    PA_CUDA(cudaEventRecord(e[i], st));
    if (i == 2) {
      for (auto& x : e) h->ev_pending.push_back(x);
      queued = true;
    }
    return PA_OK;
  }
};

// The widening pass and the attention kernel of plan P, whose sequence table
// and unit list are already on the device at d_seqs / d_units (the caller
// has sized the widened workspace for P).
int launch_plan(pa_handle h, const Plan& P, const SeqGeom* d_seqs, const Unit* d_units, int n_seq, const void* q,
                const int8_t* kp, const int8_t* vp, const float* ksc, const float* vsc, const int32_t* bt, int S,
                int W, float sm_scale, void* out, cudaStream_t st, const void* gate) {
  TimingMarks tm;
  int rc;
  if (!(rc = tm.init(h)) && !(rc = tm.mark(h, 0, st)) &&
      !(rc = launch_widen_plan(h, P, d_seqs, n_seq, kp, vp, ksc, vsc, bt, sm_scale, st)) && !(rc = tm.mark(h, 1, st)) &&
      !(rc = launch_attention_plan(h, P, d_seqs, d_units, (int)P.units.size(), q, S, W, sm_scale, out, st, gate,
                                   false, nullptr, 0, reinterpret_cast<const int*>(d_units + P.units.size()),
                                   P.n_pairs)))
    rc = tm.mark(h, 2, st);
  if (rc) tm.release(h);
  return rc;
}

int run(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const int8_t* kp, const int8_t* vp,
        const float* ksc, const float* vsc, const int32_t* bt, int S, int W, float sm_scale, void* out,
        cudaStream_t st, const void* gate = nullptr) {
  int rc = check_inputs(h, q, kp, vp, ksc, vsc, bt, out);
  if (rc) return rc;
  if (gate && !aligned(gate, 16)) return PA_EINVAL;
  if (!(sm_scale == sm_scale) || sm_scale < 0.f) return PA_EINVAL;
  if ((rc = prepare(h, n_seq, seqs, S, W, st))) return rc;
  return launch_plan(h, h->plan, h->d_seqs, h->d_units, n_seq, q, kp, vp, ksc, vsc, bt, S, W, sm_scale, out, st,
                     gate);
}

}  // namespace

extern "C" {

void pa_default_options(pa_options* opt) {
  if (!opt) return;
  opt->q_mode = PA_Q_BF16;
  opt->p_mode = PA_P_F16;
  opt->wait_timeout_ms = 2000;
  opt->record_timing = 0;
  opt->debug_stall = 0;
  opt->debug_fail_host = 0;
}

const char* pa_strerror(int code) {
  switch (code) {
    case PA_OK: return "ok";
    case PA_EINVAL: return "invalid argument";
    case PA_EARCH: return "device is not an sm_103 GPU";
    case PA_ECUDA: return "CUDA call failed";
    case PA_ETIMEOUT: return "device-side wait timed out";
    case PA_EBADPAGE: return "block-table entry outside the pool";
    case PA_ENOMEM: return "out of device memory";
    case PA_ENOSCRATCH: return "call exceeds the static scratch of pa_prefill_noalloc";
    default: return "unknown error";
  }
}

int pa_create(pa_handle* out, int n_q_heads, int n_kv_heads, int head_dim, int page_size, int n_pool_pages,
              int max_pages_per_seq, const pa_options* opt) {
  if (!out) return PA_EINVAL;
  *out = nullptr;
  if (head_dim != kHeadDim || page_size != kPage) return PA_EINVAL;
  if (n_q_heads <= 0 || n_kv_heads <= 0 || n_kv_heads > 8 || n_q_heads % n_kv_heads) return PA_EINVAL;
  const int G = n_q_heads / n_kv_heads;
  if (G > kRows || kRows % G) return PA_EINVAL;
  if (n_pool_pages <= 0 || max_pages_per_seq <= 0) return PA_EINVAL;
  pa_options o;
  pa_default_options(&o);
  if (opt) o = *opt;
  if ((o.q_mode != PA_Q_BF16 && o.q_mode != PA_Q_INT8) || (o.p_mode != PA_P_F16 && o.p_mode != PA_P_U8) ||
      o.wait_timeout_ms <= 0)
    return PA_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ECUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PA_ECUDA;
  if (prop.major != 10 || prop.minor != 3) return PA_EARCH;
  if (!encode_fn()) return PA_ECUDA;
  pa_ctx* h = new pa_ctx();
  h->HQ = n_q_heads;
  h->HKV = n_kv_heads;
  h->G = G;
  h->TQ = kRows / G;
  h->n_pool = n_pool_pages;
  h->max_pages = max_pages_per_seq;
  h->opt = o;
  h->device = dev;
  h->n_sm = prop.multiProcessorCount;
  if (cudaMalloc(&h->d_err, sizeof(int)) != cudaSuccess ||
      cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->upload_done, cudaEventDisableTiming) != cudaSuccess) {
    pa_destroy(h);
    return PA_ECUDA;
  }
  *out = h;
  return PA_OK;
}

void pa_destroy(pa_handle h) {
  if (!h) return;
  cudaDeviceSynchronize();
  void* ptrs[] = {h->kw, h->vt, h->ks, h->vs, h->vsmax, h->d_seqs, h->d_units, h->d_err, h->d_qflags, h->d_part,
                  h->d_tickets};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  for (int i = 0; i < 7; ++i)
    if (h->hb[i]) cudaFree(h->hb[i]);
  if (h->h_stage) cudaFreeHost(h->h_stage);
  if (h->upload_done) cudaEventDestroy(h->upload_done);
  for (cudaEvent_t e : h->ev_free) cudaEventDestroy(e);
  for (cudaEvent_t e : h->ev_pending) cudaEventDestroy(e);
  for (cudaEvent_t e : h->pipe_ev) cudaEventDestroy(e);
  if (h->d_pseqs) cudaFree(h->d_pseqs);
  if (h->d_punits) cudaFree(h->d_punits);
  if (h->h_pstage) cudaFreeHost(h->h_pstage);
  if (h->pstage_done) cudaEventDestroy(h->pstage_done);
  if (h->s_h2d) cudaStreamDestroy(h->s_h2d);
  if (h->s_d2h) cudaStreamDestroy(h->s_d2h);
  delete h;
}

int pa_prefill(pa_handle h, const void* q, const int8_t* k_pool, const int8_t* v_pool, const float* k_scale,
               const float* v_scale, const int32_t* block_table, int q_start, int n_q, int n_ctx, int n_sink_blk,
               int n_win_blk, float sm_scale, void* out, void* stream) {
  pa_seq s{0, q_start, n_q, n_ctx};
  return run(h, 1, &s, q, k_pool, v_pool, k_scale, v_scale, block_table, n_sink_blk, n_win_blk, sm_scale, out,
             static_cast<cudaStream_t>(stream));
}

int pa_prefill_batch(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const int8_t* k_pool,
                     const int8_t* v_pool, const float* k_scale, const float* v_scale, const int32_t* block_table,
                     int n_sink_blk, int n_win_blk, float sm_scale, void* out, void* stream) {
  return run(h, n_seq, seqs, q, k_pool, v_pool, k_scale, v_scale, block_table, n_sink_blk, n_win_blk, sm_scale, out,
             static_cast<cudaStream_t>(stream));
}

int pa_prefill_batch_gated(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const void* q_gate,
                           const int8_t* k_pool, const int8_t* v_pool, const float* k_scale, const float* v_scale,
                           const int32_t* block_table, int n_sink_blk, int n_win_blk, float sm_scale, void* out,
                           void* stream) {
  if (!q_gate) return PA_EINVAL;
  return run(h, n_seq, seqs, q, k_pool, v_pool, k_scale, v_scale, block_table, n_sink_blk, n_win_blk, sm_scale, out,
             static_cast<cudaStream_t>(stream), q_gate);
}

// A piece of a sequence's query rows, computed as one call of its own.
// The host-buffer path is a pipeline over chunks of the query rows: the pool,
// scales and block table go in first and are widened once, then each chunk's
// q rows go in on one copy stream while the previous chunk is computed on the
// caller's stream and the one before that is copied out on another copy
// stream.  A chunk is a contiguous run of the sequences' rows laid end to
// end; a chunk boundary inside a sequence falls on a multiple of a work
// unit's tokens (256 / G, units start on those multiples), so every unit of
// the call's one plan belongs to exactly one chunk, and a chunk's attention
// launch runs just its units.
int pa_prefill_host(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const int8_t* k_pool,
                    const int8_t* v_pool, const float* k_scale, const float* v_scale, const int32_t* block_table,
                    int n_sink_blk, int n_win_blk, float sm_scale, void* out, void* stream) {
  if (!h || n_seq <= 0 || !seqs) return PA_EINVAL;
  // the whole call's plan validates it and sizes the widened workspace once
  Plan whole;
  int rc = build_plan(h->HQ, h->HKV, n_seq, seqs, n_sink_blk, n_win_blk, h->max_pages, whole);
  if (rc) return rc;
  const int total_q = whole.total_q;
  const size_t row_bytes = (size_t)h->HQ * kHeadDim * 2;  // one token's q (or out) row
  const size_t bytes[7] = {
      (size_t)total_q * row_bytes,                           // q
      (size_t)h->n_pool * kPage * h->HKV * kHeadDim,          // k_pool
      (size_t)h->n_pool * kPage * h->HKV * kHeadDim,          // v_pool
      (size_t)h->n_pool * kPage * h->HKV * sizeof(float),     // k_scale
      (size_t)h->n_pool * kPage * h->HKV * sizeof(float),     // v_scale
      (size_t)n_seq * h->max_pages * sizeof(int32_t),         // block table
      (size_t)total_q * row_bytes};                           // out
  const void* src[6] = {q, k_pool, v_pool, k_scale, v_scale, block_table};
  for (int i = 0; i < 6; ++i)
    if (!src[i]) return PA_EINVAL;
  if (!out) return PA_EINVAL;
  if (!(sm_scale == sm_scale) || sm_scale < 0.f) return PA_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < 7; ++i)
    if ((rc = grow_bytes(h->hb[i], h->hb_cap[i], bytes[i]))) return rc;

  // chunk boundaries on the sequences' rows laid end to end
  std::vector<long long> base(n_seq + 1, 0);  // first row of each sequence, end to end
  for (int s = 0; s < n_seq; ++s) base[s + 1] = base[s] + seqs[s].n_q;
  std::vector<long long> cuts;
  if ((rc = host_chunk_ends(h->HQ, h->HKV, n_seq, seqs, pa::attention_pairs(h->n_sm), cuts))) return rc;
  std::vector<std::vector<pa_seq>> chunks;  // per chunk, its pieces of the sequences (rows, same context)
  std::vector<long long> ends;  // chunk ends, end to end
  long long lo = 0;
  for (const long long hi : cuts) {
    if (hi <= lo) continue;
    chunks.emplace_back();
    ends.push_back(hi);
    for (int s = 0; s < n_seq; ++s) {
      const long long a = std::max(lo, base[s]), b = std::min(hi, base[s + 1]);
      if (a >= b) continue;
      const int qa = seqs[s].q_start + (int)(a - base[s]);
      chunks.back().push_back(pa_seq{seqs[s].q_off + (qa - seqs[s].q_start), qa, (int)(b - a), seqs[s].n_ctx});
    }
    lo = hi;
  }
  const int n_ch = (int)chunks.size();

  // one plan for the whole call (so one widening pass and the same per-sequence
  // V-scale maximum as pa_prefill_batch); its units split by chunk, each
  // chunk's list still in decreasing cost; all uploaded in one go ahead of the
  // large copies (a small copy queued behind them would hold up the first chunk)
  Plan P;
  if ((rc = build_plan(h->HQ, h->HKV, n_seq, seqs, n_sink_blk, n_win_blk, h->max_pages, P))) return rc;
  std::vector<std::vector<Unit>> cunits(n_ch);
  for (const Unit& u : P.units) {
    const pa_seq& q0 = seqs[u.seq];
    const long long row = base[u.seq] + (std::max(u.t0, q0.q_start) - q0.q_start);  // its first row, end to end
    const int c = (int)(std::upper_bound(ends.begin(), ends.end(), row) - ends.begin());
    if (c >= n_ch) return PA_EINVAL;  // cannot happen: every row lies in a chunk
    cunits[c].push_back(u);
  }
  // each chunk's units laid out pair by pair for its launch's pairs, the pair
  // offsets after them
  std::vector<std::vector<int>> coff(n_ch);
  std::vector<int> cpairs(n_ch, 0);
  std::vector<size_t> off_u(n_ch);
  size_t n_u = 0;
  for (int c = 0; c < n_ch; ++c) {
    const int n = (int)cunits[c].size();
    cpairs[c] = launch_pairs(h->n_sm, n);
    std::vector<Unit> by_pair;
    assign_pairs(cunits[c].data(), n, cpairs[c], by_pair, coff[c]);
    cunits[c] = std::move(by_pair);
    off_u[c] = n_u;
    n_u += (size_t)n + pair_off_records(cpairs[c]);
  }
  const size_t n_s = P.seqs.size();
  if ((rc = reserve_rows(h, (size_t)P.n_tok_total))) return rc;
  if ((rc = grow(h->vsmax, h->vsmax_cap, (size_t)n_seq * h->HKV))) return rc;
  if ((rc = grow(h->d_pseqs, h->pseqs_cap, n_s))) return rc;
  if ((rc = grow(h->d_punits, h->punits_cap, n_u))) return rc;
  if (!h->pstage_done) PA_CUDA(cudaEventCreateWithFlags(&h->pstage_done, cudaEventDisableTiming));
  if (h->pstage_recorded) PA_CUDA(cudaEventSynchronize(h->pstage_done));  // staging free again
  const size_t bytes_s = n_s * sizeof(SeqGeom), bytes_u = n_u * sizeof(Unit);
  if (h->h_pstage_cap < bytes_s + bytes_u) {
    if (h->h_pstage) cudaFreeHost(h->h_pstage);
    h->h_pstage = nullptr;
    h->h_pstage_cap = 0;
    PA_CUDA(cudaMallocHost(&h->h_pstage, bytes_s + bytes_u));
    h->h_pstage_cap = bytes_s + bytes_u;
  }
  std::memcpy(h->h_pstage, P.seqs.data(), bytes_s);
  for (int c = 0; c < n_ch; ++c) {
    Unit* dst = reinterpret_cast<Unit*>(static_cast<char*>(h->h_pstage) + bytes_s) + off_u[c];
    std::memcpy(dst, cunits[c].data(), cunits[c].size() * sizeof(Unit));
    std::memcpy(dst + cunits[c].size(), coff[c].data(), coff[c].size() * sizeof(int));
  }
  PA_CUDA(cudaMemcpyAsync(h->d_pseqs, h->h_pstage, bytes_s, cudaMemcpyHostToDevice, st));
  PA_CUDA(cudaMemcpyAsync(h->d_punits, static_cast<char*>(h->h_pstage) + bytes_s, bytes_u, cudaMemcpyHostToDevice, st));
  PA_CUDA(cudaEventRecord(h->pstage_done, st));
  h->pstage_recorded = true;

  // chunk c > 0 waits for its rows on the device (a flag the copy stream
  // writes after them), not with an event wait on the stream, so that its
  // launch can overlap the previous chunk's (programmatic dependent launch)
  const WriteValue32Fn write_value = write_value_fn();
  if (write_value && h->qflags_cap < n_ch) {
    if (h->d_qflags) cudaFree(h->d_qflags);
    h->d_qflags = nullptr;
    h->qflags_cap = 0;
    PA_CUDA(cudaMalloc(&h->d_qflags, (size_t)n_ch * sizeof(unsigned int)));
    PA_CUDA(cudaMemset(h->d_qflags, 0, (size_t)n_ch * sizeof(unsigned int)));
    h->qflags_cap = n_ch;
  }
  if (++h->q_epoch == 0) h->q_epoch = 1;  // flags start at 0: never a live epoch
  const unsigned int epoch = h->q_epoch;

  // streams and events
  if (!h->s_h2d) PA_CUDA(cudaStreamCreateWithFlags(&h->s_h2d, cudaStreamNonBlocking));
  if (!h->s_d2h) PA_CUDA(cudaStreamCreateWithFlags(&h->s_d2h, cudaStreamNonBlocking));
  const size_t n_ev = 3 + 2 * (size_t)n_ch;
  while (h->pipe_ev.size() < n_ev) {
    cudaEvent_t e;
    PA_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    h->pipe_ev.push_back(e);
  }
  cudaEvent_t ev_start = h->pipe_ev[0], ev_end = h->pipe_ev[1], ev_pool = h->pipe_ev[2];
  cudaEvent_t* ev_in = h->pipe_ev.data() + 3;           // chunk c's q rows are in
  cudaEvent_t* ev_done = h->pipe_ev.data() + 3 + n_ch;  // chunk c is computed

  // From the first copy on, the caller's host buffers are in use by copies on
  // the handle's streams: on any failure the call drains those streams (and
  // `stream`) before it returns, so no copy still reads q or the pool, or
  // writes out, once the caller gets control back.  Every chunk's row flag is
  // written before the first chunk launch, so the drain always ends.
  TimingMarks tm;
  auto enqueue = [&]() -> int {
    // inputs: after whatever the caller's stream did before
    PA_CUDA(cudaEventRecord(ev_start, st));
    PA_CUDA(cudaStreamWaitEvent(h->s_h2d, ev_start, 0));
    for (int i = 1; i < 6; ++i) PA_CUDA(cudaMemcpyAsync(h->hb[i], src[i], bytes[i], cudaMemcpyHostToDevice, h->s_h2d));
    PA_CUDA(cudaEventRecord(ev_pool, h->s_h2d));
    for (int c = 0; c < n_ch; ++c) {
      for (const pa_seq& pc : chunks[c]) {
        const size_t off = (size_t)pc.q_off * row_bytes;
        PA_CUDA(cudaMemcpyAsync(static_cast<char*>(h->hb[0]) + off, static_cast<const char*>(q) + off,
                                (size_t)pc.n_q * row_bytes, cudaMemcpyHostToDevice, h->s_h2d));
      }
      PA_CUDA(cudaEventRecord(ev_in[c], h->s_h2d));
      // test hook: a failure of the enqueue after the pool and the first rows are in flight
      if (h->opt.debug_fail_host && c == std::min(1, n_ch - 1)) return PA_ECUDA;
      if (write_value && c > 0 &&
          write_value(h->s_h2d, (CUdeviceptr)(h->d_qflags + c), epoch, CU_STREAM_WRITE_VALUE_DEFAULT) != CUDA_SUCCESS)
        return PA_ECUDA;
    }
    // widen the whole pool once it is in, then compute each chunk once its rows
    // are in; copy its output out behind it
    PA_CUDA(cudaStreamWaitEvent(h->s_d2h, ev_start, 0));
    PA_CUDA(cudaStreamWaitEvent(st, ev_pool, 0));
    int r = PA_OK;
    if (!(r = tm.init(h)) && !(r = tm.mark(h, 0, st)))
      r = launch_widen_plan(h, P, h->d_pseqs, n_seq, static_cast<const int8_t*>(h->hb[1]),
                            static_cast<const int8_t*>(h->hb[2]), static_cast<const float*>(h->hb[3]),
                            static_cast<const float*>(h->hb[4]), static_cast<const int32_t*>(h->hb[5]), sm_scale, st);
    if (!r) r = tm.mark(h, 1, st);
    if (r) return r;
    bool after_attn = false;  // the last launch on st is an attention launch of this call
    for (int c = 0; c < n_ch; ++c) {
      const bool on_device = write_value && c > 0 && after_attn;
      if (!on_device) PA_CUDA(cudaStreamWaitEvent(st, ev_in[c], 0));
      if (!cunits[c].empty()) {
        if ((r = launch_attention_plan(h, P, h->d_pseqs, h->d_punits + off_u[c], (int)cunits[c].size(), h->hb[0],
                                       n_sink_blk, n_win_blk, sm_scale, h->hb[6], st, nullptr, on_device,
                                       on_device ? h->d_qflags + c : nullptr, epoch,
                                       reinterpret_cast<const int*>(h->d_punits + off_u[c] + cunits[c].size()),
                                       cpairs[c])))
          return r;
        after_attn = true;
      }
      PA_CUDA(cudaEventRecord(ev_done[c], st));
      PA_CUDA(cudaStreamWaitEvent(h->s_d2h, ev_done[c], 0));
      for (const pa_seq& pc : chunks[c]) {
        const size_t off = (size_t)pc.q_off * row_bytes;
        PA_CUDA(cudaMemcpyAsync(static_cast<char*>(out) + off, static_cast<const char*>(h->hb[6]) + off,
                                (size_t)pc.n_q * row_bytes, cudaMemcpyDeviceToHost, h->s_d2h));
      }
    }
    if ((r = tm.mark(h, 2, st))) return r;
    // the caller's stream waits for both copy streams
    PA_CUDA(cudaEventRecord(ev_end, h->s_d2h));
    PA_CUDA(cudaStreamWaitEvent(st, ev_end, 0));
    PA_CUDA(cudaEventRecord(ev_start, h->s_h2d));
    PA_CUDA(cudaStreamWaitEvent(st, ev_start, 0));
    return PA_OK;
  };
  if ((rc = enqueue())) {
    tm.release(h);
    // errors of the drain itself are ignored: the first failure is reported
    (void)cudaStreamSynchronize(h->s_h2d);
    (void)cudaStreamSynchronize(h->s_d2h);
    (void)cudaStreamSynchronize(st);
    return rc;
  }
  return pa_last_error(h, stream);
}

int pa_debug_copy_streams_idle(pa_handle h) {
  if (!h) return PA_EINVAL;
  for (cudaStream_t s : {h->s_h2d, h->s_d2h}) {
    if (!s) continue;
    const cudaError_t e = cudaStreamQuery(s);
    if (e == cudaErrorNotReady) return 0;
    if (e != cudaSuccess) return PA_ECUDA;
  }
  return 1;
}

int pa_last_error(pa_handle h, void* stream) {
  if (!h) return PA_EINVAL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ECUDA;
  int e = 0;
  if (cudaMemcpy(&e, h->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ECUDA;
  if (e != 0 && cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess) return PA_ECUDA;
  if (e & DEV_ERR_TIMEOUT) return PA_ETIMEOUT;
  if (e & DEV_ERR_BAD_PAGE) return PA_EBADPAGE;
  if (e != 0) return PA_ECUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}

int pa_timing(pa_handle h, int reset, double* widen_ms, double* attention_ms, int* n_calls) {
  if (!h) return PA_EINVAL;
  for (size_t i = 0; i + 2 < h->ev_pending.size(); i += 3) {
    cudaEvent_t* e = &h->ev_pending[i];
    if (cudaEventSynchronize(e[2]) != cudaSuccess) return PA_ECUDA;
    float a = 0.f, b = 0.f;
    cudaEventElapsedTime(&a, e[0], e[1]);
    cudaEventElapsedTime(&b, e[1], e[2]);
    h->t_widen += a;
    h->t_attn += b;
    h->t_calls += 1;
    for (int k = 0; k < 3; ++k) h->ev_free.push_back(e[k]);
  }
  h->ev_pending.clear();
  if (widen_ms) *widen_ms = h->t_widen;
  if (attention_ms) *attention_ms = h->t_attn;
  if (n_calls) *n_calls = h->t_calls;
  if (reset) {
    h->t_widen = h->t_attn = 0.0;
    h->t_calls = 0;
  }
  return PA_OK;
}

int pa_plan(int n_q_heads, int n_kv_heads, int n_seq, const pa_seq* seqs, int n_sink_blk, int n_win_blk,
            int32_t* units_out, int cap, int* n_units, long long* n_tiles, int* n_widened_rows) {
  Plan P;
  int rc = build_plan(n_q_heads, n_kv_heads, n_seq, seqs, n_sink_blk, n_win_blk, 0, P);
  if (rc) return rc;
  if (n_units) *n_units = (int)P.units.size();
  if (n_tiles) *n_tiles = P.n_tiles;
  if (n_widened_rows) *n_widened_rows = P.n_tok_total;
  if (units_out) {
    const int n = std::min(cap, (int)P.units.size());
    for (int i = 0; i < n; ++i) {
      units_out[4 * i + 0] = P.units[i].seq;
      units_out[4 * i + 1] = P.units[i].g;
      units_out[4 * i + 2] = P.units[i].t0;
      units_out[4 * i + 3] = P.units[i].n_tiles;
    }
  }
  return PA_OK;
}

int pa_plan_pairs(int n_q_heads, int n_kv_heads, int n_seq, const pa_seq* seqs, int n_sink_blk, int n_win_blk,
                  int n_pairs, int32_t* units_out, int cap, int32_t* pair_off, int* n_units) {
  if (n_pairs < 1 || !pair_off) return PA_EINVAL;
  Plan P;
  int rc = build_plan(n_q_heads, n_kv_heads, n_seq, seqs, n_sink_blk, n_win_blk, 0, P);
  if (rc) return rc;
  const int n = (int)P.units.size();
  if (n_units) *n_units = n;
  if (units_out && cap < n) return PA_EINVAL;
  std::vector<Unit> by_pair;
  std::vector<int> off;
  assign_pairs(P.units.data(), n, n_pairs, by_pair, off);
  std::copy(off.begin(), off.end(), pair_off);
  if (units_out)
    for (int i = 0; i < n; ++i) {
      units_out[4 * i + 0] = by_pair[(size_t)i].seq;
      units_out[4 * i + 1] = by_pair[(size_t)i].g;
      units_out[4 * i + 2] = by_pair[(size_t)i].t0;
      units_out[4 * i + 3] = by_pair[(size_t)i].n_tiles;
    }
  return PA_OK;
}

int pa_host_chunks(int n_q_heads, int n_kv_heads, int n_seq, const pa_seq* seqs, int n_pairs, long long* chunk_end,
                   int cap, int* n_chunks) {
  std::vector<long long> ends;
  const int rc = host_chunk_ends(n_q_heads, n_kv_heads, n_seq, seqs, n_pairs, ends);
  if (rc) return rc;
  if (n_chunks) *n_chunks = (int)ends.size();
  if (chunk_end) {
    if ((int)ends.size() > cap) return PA_EINVAL;
    std::copy(ends.begin(), ends.end(), chunk_end);
  }
  return PA_OK;
}

int pa_debug_gather(pa_handle h, int n_seq, const pa_seq* seqs, const int8_t* k_pool, const int8_t* v_pool,
                    const float* k_scale, const float* v_scale, const int32_t* block_table, int n_sink_blk,
                    int n_win_blk, int seq, int8_t* k_out, int8_t* v_out, float* ks_out, float* vs_out,
                    int32_t* tok_out, int cap, int* n_rows, void* stream) {
  if (!h || !k_out || !v_out || !ks_out || !vs_out || !tok_out || !n_rows || seq < 0 || seq >= n_seq)
    return PA_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = prepare(h, n_seq, seqs, n_sink_blk, n_win_blk, st);
  if (rc) return rc;
  const int rows = h->plan.seqs[seq].n_blocks * kPage;
  *n_rows = rows;
  if (rows > cap) return PA_EINVAL;
  PA_CUDA(cudaMemsetAsync(h->vsmax, 0, sizeof(unsigned int) * n_seq * h->HKV, st));
  PA_CUDA(launch_widen(widen_params(h, k_pool, v_pool, k_scale, v_scale, block_table, n_seq), st));
  PA_CUDA(launch_debug_gather(widen_params(h, k_pool, v_pool, k_scale, v_scale, block_table, n_seq), seq, k_out,
                              v_out, ks_out, vs_out, tok_out, st));
  return pa_last_error(h, stream);
}

int pa_debug_qcodes(const void* q_rows, int n_rows, int8_t* codes, float* scales, void* stream) {
  if (n_rows < 0 || (n_rows > 0 && (!q_rows || !codes || !scales))) return PA_EINVAL;
  if (n_rows == 0) return PA_OK;
  if (!aligned(q_rows, 16) || !aligned(codes, 4) || !aligned(scales, 4)) return PA_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PA_CUDA(launch_debug_qcodes(static_cast<const __nv_bfloat16*>(q_rows), n_rows, codes, scales, st));
  PA_CUDA(cudaStreamSynchronize(st));
  return PA_OK;
}

int pa_kv_append(pa_handle h, const void* k_new, const void* v_new, int n_new, int tok_start,
                 const int32_t* block_table_row, int8_t* k_pool, int8_t* v_pool, float* k_scale, float* v_scale,
                 void* stream) {
  if (!h || n_new < 0 || tok_start < 0) return PA_EINVAL;
  if (n_new == 0) return PA_OK;
  if (!k_new || !v_new || !block_table_row || !k_pool || !v_pool || !k_scale || !v_scale) return PA_EINVAL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(block_table_row, 4))
    return PA_EINVAL;
  if ((long long)tok_start + n_new > (long long)h->max_pages * kPage) return PA_EINVAL;
  KvAppendParams p{};
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.n_new = n_new;
  p.tok_start = tok_start;
  p.HKV = h->HKV;
  p.n_pool = h->n_pool;
  p.bt_row = block_table_row;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err = h->d_err;
  PA_CUDA(launch_kv_append(p, static_cast<cudaStream_t>(stream)));
  return PA_OK;
}

namespace {
// Cost-balanced decode runs over a launch's pair list (block counts `len`,
// HKV pairs per sequence).  A CTA costs its blocks plus kDecSegCost for every
// pair after its first: a run that crosses into another pair waits for all
// its warps, combines them, loads the next pair's query rows and refills its
// copies (measured at 64 sequences x 32k context: such CTAs ended ~10 us,
// about 16 blocks' worth, after the others).  Greedy packing under `budget`;
// false if it needs more than max_ctas CTAs.
constexpr int kDecSegCost = 16;
bool decode_pack(const std::vector<int>& len, int HKV, long long total, long long budget, long long max_ctas,
                 DecRuns& r) {
  r.x0.clear();
  r.seq.clear();
  r.slot.clear();
  r.max_slots = 1;
  std::vector<int> first_cta(len.size(), 0);
  size_t pi = 0;
  long long pstart = 0, x = 0;
  int cta = 0;
  while (x < total) {
    if (cta >= max_ctas) return false;
    r.x0.push_back((int)x);
    r.seq.push_back((int)(pi / (size_t)HKV));
    r.slot.push_back(x == pstart ? 0 : cta - first_cta[pi]);
    long long cost = 0;
    bool first = true;
    while (x < total) {
      const long long pend = pstart + len[pi];
      const long long extra = first ? 0 : kDecSegCost;
      if (cost + extra >= budget) break;
      if (x == pstart) first_cta[pi] = cta;
      const long long take = std::min(pend - x, budget - cost - extra);
      cost += extra + take;
      x += take;
      first = false;
      if (x < pend) break;  // the budget ran out inside the pair
      r.max_slots = std::max(r.max_slots, cta - first_cta[pi] + 1);
      ++pi;
      pstart = pend;
    }
    ++cta;
  }
  return true;
}

// Visible blocks of a decode query (the context's last token, t = n_ctx - 1)
// under the prefill's block mask: sink blocks, then the window run up to t's block.
int decode_n_vis(int n_ctx, int n_sink_blk, int n_win_blk) {
  const int last = (n_ctx - 1) / kPage;
  const int lo = n_win_blk > 0 ? std::max(0, last + 1 - n_win_blk) : 0;
  const int n_sink = n_win_blk > 0 ? std::min(std::max(n_sink_blk, 0), lo) : 0;
  return n_sink + (last - lo + 1);
}

// One decode launch (up to kDecParamSeqs sequences): the launch's pairs'
// blocks end to end; one wave of cost-balanced runs listed in the parameters
// when runs of at most 128 blocks fit in one wave, else whole waves of equal
// runs of per_cta blocks.
struct DecLaunch {
  int s0 = 0, n = 0, total = 0, per_cta = 0, n_cta = 0, max_slots = 1;
  bool listed = false;
  DecRuns runs;
};
int decode_launch_plan(int HKV, long long slots, const int* n_vis, int s0, int n, DecLaunch& L) {
  L = DecLaunch{};
  L.s0 = s0;
  L.n = n;
  long long vis = 0;
  int nv_max = 1;
  std::vector<int> len;
  for (int i = 0; i < n; ++i) {
    vis += n_vis[i];
    nv_max = std::max(nv_max, n_vis[i]);
    for (int g = 0; g < HKV; ++g) len.push_back(n_vis[i]);
  }
  const long long total = vis * HKV;
  if (total >= (1ll << 30) || slots < 1) return PA_EINVAL;
  L.total = (int)total;
  const long long wave = std::min<long long>(slots, kDecParamCtas);
  if (total <= wave * kDecMaxCtaBlocks && decode_pack(len, HKV, total, kDecMaxCtaBlocks, wave, L.runs)) {
    long long lo = std::max(1ll, (total + wave - 1) / wave), hi = kDecMaxCtaBlocks;
    while (lo < hi) {  // the smallest budget that packs into one wave
      const long long mid = (lo + hi) / 2;
      if (decode_pack(len, HKV, total, mid, wave, L.runs)) hi = mid;
      else lo = mid + 1;
    }
    (void)decode_pack(len, HKV, total, lo, wave, L.runs);
    L.listed = true;
    L.per_cta = (int)lo;
    L.n_cta = (int)L.runs.x0.size();
    L.max_slots = L.runs.max_slots;
  } else {
    const long long full = (total + kDecMaxCtaBlocks - 1) / kDecMaxCtaBlocks;
    const long long waves = std::max(1ll, (full + slots - 1) / slots);
    L.listed = false;
    L.per_cta = (int)std::max(1ll, (total + waves * slots - 1) / (waves * slots));
    L.n_cta = (int)((total + L.per_cta - 1) / L.per_cta);
    L.max_slots = (nv_max - 1 + L.per_cta - 1) / L.per_cta + 1;  // CTA runs a pair's blocks can meet
  }
  return PA_OK;
}

// A decode query's checks: one token, the context's last, within the block table.
bool decode_seq_ok(const pa_seq& q1, int max_pages) {
  return q1.n_q == 1 && q1.q_off >= 0 && q1.n_ctx >= 1 && q1.q_start == q1.n_ctx - 1 &&
         (q1.n_ctx + kPage - 1) / kPage <= max_pages;
}
}  // namespace

int pa_decode_plan(int n_kv_heads, int slots, int n_seq, const pa_seq* seqs, int n_sink_blk, int n_win_blk,
                   int32_t* runs_out, int cap, int* n_cta, int* per_cta, int* max_slots, int* listed,
                   long long* total_blocks) {
  if (n_kv_heads < 1 || n_kv_heads > 8 || slots < 1 || n_seq <= 0 || !seqs) return PA_EINVAL;
  const int n = std::min(n_seq, kDecParamSeqs);
  std::vector<int> n_vis((size_t)n);
  for (int s = 0; s < n; ++s) {
    if (!decode_seq_ok(seqs[s], INT32_MAX)) return PA_EINVAL;
    n_vis[(size_t)s] = decode_n_vis(seqs[s].n_ctx, n_sink_blk, n_win_blk);
  }
  DecLaunch L;
  const int rc = decode_launch_plan(n_kv_heads, slots, n_vis.data(), 0, n, L);
  if (rc) return rc;
  if (n_cta) *n_cta = L.n_cta;
  if (per_cta) *per_cta = L.per_cta;
  if (max_slots) *max_slots = L.max_slots;
  if (listed) *listed = L.listed ? 1 : 0;
  if (total_blocks) *total_blocks = L.total;
  if (runs_out) {
    if (cap < L.n_cta) return PA_EINVAL;
    if (L.listed) {
      for (int c = 0; c < L.n_cta; ++c) {
        runs_out[3 * c] = L.runs.x0[(size_t)c];
        runs_out[3 * c + 1] = L.runs.seq[(size_t)c];
        runs_out[3 * c + 2] = L.runs.slot[(size_t)c];
      }
    } else {  // equal runs: CTA c starts at c per_cta; its slot counts the CTAs before it in that block's pair
      long long pstart = 0;
      int s = 0, g = 0;
      for (int c = 0; c < L.n_cta; ++c) {
        const long long x = (long long)c * L.per_cta;
        while (x >= pstart + n_vis[(size_t)s]) {
          pstart += n_vis[(size_t)s];
          if (++g == n_kv_heads) {
            g = 0;
            ++s;
          }
        }
        runs_out[3 * c] = (int)x;
        runs_out[3 * c + 1] = s;
        runs_out[3 * c + 2] = c - (int)(pstart / L.per_cta);
      }
    }
  }
  return PA_OK;
}

int pa_decode(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const int8_t* k_pool, const int8_t* v_pool,
              const float* k_scale, const float* v_scale, const int32_t* block_table, int n_sink_blk, int n_win_blk,
              float sm_scale, void* out, void* stream) {
  int rc = check_inputs(h, q, k_pool, v_pool, k_scale, v_scale, block_table, out);
  if (rc) return rc;
  if (n_seq <= 0 || !seqs || h->G > 8 || !(sm_scale == sm_scale) || sm_scale < 0.f) return PA_EINVAL;
  std::vector<int> n_vis((size_t)n_seq);
  for (int s = 0; s < n_seq; ++s) {
    if (!decode_seq_ok(seqs[s], h->max_pages)) return PA_EINVAL;
    n_vis[(size_t)s] = decode_n_vis(seqs[s].n_ctx, n_sink_blk, n_win_blk);
  }
  // launches of up to kDecParamSeqs sequences, their table in the launch's parameters
  std::vector<DecLaunch> launches;
  const long long slots = (long long)h->n_sm * decode_ctas_per_sm(h->HKV);
  size_t part_need = 0;
  for (int s0 = 0; s0 < n_seq; s0 += kDecParamSeqs) {
    DecLaunch L;
    if ((rc = decode_launch_plan(h->HKV, slots, n_vis.data() + s0, s0, std::min(kDecParamSeqs, n_seq - s0), L)))
      return rc;
    part_need = std::max(part_need, (size_t)L.n * h->HKV * L.max_slots * h->G * kDecPartStride);
    launches.push_back(std::move(L));
  }
  if (part_need > (size_t)INT32_MAX) return PA_EINVAL;
  if ((rc = grow(h->d_part, h->part_cap, part_need))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->tickets_cap < kDecParamSeqs * h->HKV) {
    if ((rc = grow(h->d_tickets, h->tickets_cap, (size_t)kDecParamSeqs * h->HKV))) return rc;
    PA_CUDA(cudaMemsetAsync(h->d_tickets, 0, (size_t)h->tickets_cap * sizeof(unsigned long long), st));
  }
  if (k_pool != h->dec_kp || v_pool != h->dec_vp) {
    // the pool as uint8 [n_pool * 16][HKV][256]; a box is one kv head's 16 token rows of half the dims
    const uint64_t dims[3] = {(uint64_t)kHeadDim, (uint64_t)h->HKV, (uint64_t)h->n_pool * kPage};
    const uint64_t strides[2] = {(uint64_t)kHeadDim, (uint64_t)h->HKV * kHeadDim};
    const uint32_t box[3] = {128, 1, (uint32_t)kPage};
    h->dec_kp = h->dec_vp = nullptr;
    if ((rc = encode(&h->dec_maps.k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, k_pool, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B)) ||
        (rc = encode(&h->dec_maps.v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, v_pool, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B)))
      return rc;
    h->dec_kp = k_pool;
    h->dec_vp = v_pool;
  }
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_table = block_table;
  p.bt_stride = h->max_pages;
  p.n_pool = h->n_pool;
  p.S = n_sink_blk;
  p.W = n_win_blk;
  p.HQ = h->HQ;
  p.HKV = h->HKV;
  p.G = h->G;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.part = h->d_part;
  p.tickets = h->d_tickets;
  p.err = h->d_err;
  p.wait_ns = (unsigned long long)h->opt.wait_timeout_ms * 1000000ull;
  DecodeSeqs tab;
  for (const DecLaunch& L : launches) {
    int vstart = 0;
    for (int i = 0; i < L.n; ++i) {
      const pa_seq& q1 = seqs[L.s0 + i];
      tab.seq[i] = make_int4(q1.q_off, q1.n_ctx, vstart, 0);
      vstart += n_vis[(size_t)(L.s0 + i)];
    }
    p.n_seq = L.n;
    p.bt_row0 = L.s0;
    p.total = L.total;
    p.per_cta = L.per_cta;
    p.max_slots = L.max_slots;
    p.runs_listed = L.listed ? 1 : 0;
    if (L.listed)
      for (int c = 0; c < L.n_cta; ++c) {
        tab.cta_x0[c] = L.runs.x0[(size_t)c];
        tab.cta_seq[c] = (uint16_t)L.runs.seq[(size_t)c];
        tab.cta_slot[c] = (uint16_t)L.runs.slot[(size_t)c];
      }
    PA_CUDA(launch_decode(p, tab, h->dec_maps, L.n_cta, st));
  }
  return PA_OK;
}

int pa_debug_maskset(pa_handle h, int n_seq, const pa_seq* seqs, int n_sink_blk, int n_win_blk,
                     int32_t* row_counts, int32_t* unit_blocks, int cap, int32_t* units_out, int units_cap,
                     int* n_units, void* stream) {
  if (!h || !row_counts || !unit_blocks || !units_out || !n_units || cap <= 0) return PA_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = prepare(h, n_seq, seqs, n_sink_blk, n_win_blk, st);
  if (rc) return rc;
  const Plan& P = h->plan;
  *n_units = (int)P.units.size();
  if ((int)P.units.size() > units_cap) return PA_EINVAL;
  for (size_t i = 0; i < P.units.size(); ++i) {
    units_out[4 * i + 0] = P.units[i].seq;
    units_out[4 * i + 1] = P.units[i].g;
    units_out[4 * i + 2] = P.units[i].t0;
    units_out[4 * i + 3] = P.units[i].n_tiles;
  }
  PA_CUDA(launch_debug_maskset(h->d_seqs, h->d_units, (int)P.units.size(), 2 * h->TQ, h->G, n_sink_blk, n_win_blk,
                               row_counts, unit_blocks, cap, st));
  return pa_last_error(h, stream);
}

}  // extern "C"
