// Allocation-free entry point: the same widening and attention kernels as
// pa_prefill, with every piece of scratch memory (widened K/V, scales, work
// list, error word) carved out of one file-scope device array instead of a
// handle's cudaMalloc'd workspace.
//
// Who needs it: callers that may not call cudaMalloc / cudaFree at all, for
// example an engine that has reserved nearly all device memory for its own
// KV-cache pool and accounts for every byte, or code on a latency-critical
// path where an allocation (which can synchronise the device) is not allowed.
// They pass inputs and outputs; this file allocates nothing.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

using namespace pa;

namespace {

// The scratch every call shares.  Each GPU that loads the library holds it
// until the process exits.  Host code must not use the symbol as an address:
// the device address comes from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr size_t kHeaderBytes = 4096;            // error word, V-scale maxima, sequence geometry
constexpr size_t kUnitsBytes = 1u << 20;         // work list
constexpr int kMaxUnits = (int)(kUnitsBytes / sizeof(Unit));
constexpr size_t kWidenedOffset = kHeaderBytes + kUnitsBytes;
// First tokens of units (one per UT query tokens) the ordering kernel ranks in
// shared memory; the widened-row limit keeps every call below it.
constexpr int kMaxT0 = 16384;
constexpr int kPlanThreads = 256;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

// Per device: the scratch's device address and the attributes a call needs,
// looked up once with that device current, and again if the device's context
// was replaced since (a reset reloads the module, which may move the array).
struct DeviceSetup {
  unsigned long long ctx_id = 0;  // unique id of the context the entry was made in (0: none yet)
  void* addr = nullptr;
  int n_sm = 0;
  bool sm103 = false;
};

int device_setup(int device, DeviceSetup* out) {
  static std::mutex mu;
  static DeviceSetup table[64];
  static CtxGetCurrentFn get_ctx = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  if (device < 0 || device >= 64 || !get_ctx || !get_id) return PA_ECUDA;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return PA_ECUDA;
  if (!ctx) {  // no context current yet: cudaSetDevice makes the device's primary context current
    if (cudaSetDevice(device) != cudaSuccess || get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return PA_ECUDA;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return PA_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  DeviceSetup& e = table[device];
  if (e.ctx_id != id || !e.addr) {
    DeviceSetup n;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.n_sm, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
      return PA_ECUDA;
    n.sm103 = major == 10 && minor == 3;
    if (n.sm103 && (cudaGetSymbolAddress(&n.addr, g_noalloc_scratch) != cudaSuccess || !n.addr)) return PA_ECUDA;
    n.ctx_id = id;
    e = n;
  }
  *out = e;
  return PA_OK;
}

// The work list in the handle planner's order: units by decreasing key tiles,
// ties by increasing first token, then kv head (a stable sort of the list
// made in token order).  For one sequence every kv head of a first token has
// the same tiles, so each first token t0_i = t_first + i UT is ranked among
// all n_t0 of them (tiles held in shared memory) and its HKV units take
// consecutive places.  Also writes the sequence geometry and clears the
// words that must start at zero.
__global__ void __launch_bounds__(kPlanThreads) noalloc_plan_kernel(SeqGeom sg, int S, int W, int HKV, int UT,
                                                                    int n_t0, int t_first, SeqGeom* seq_out,
                                                                    Unit* units, unsigned int* vsmax, int* err) {
  __shared__ uint16_t tiles[kMaxT0];
  for (int j = threadIdx.x; j < n_t0; j += kPlanThreads)
    tiles[j] = (uint16_t)unit_geom(t_first + j * UT, UT, sg, S, W).n_tiles;
  __syncthreads();
  const int i = blockIdx.x * kPlanThreads + threadIdx.x;
  if (i < n_t0) {
    const int ti = tiles[i];
    int rank = 0;
    for (int j = 0; j < n_t0; ++j) {
      const int tj = tiles[j];
      rank += (tj > ti || (tj == ti && j < i)) ? 1 : 0;
    }
    for (int g = 0; g < HKV; ++g) units[rank * HKV + g] = Unit{0, g, t_first + i * UT, ti};
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *seq_out = sg;
    *err = 0;
  }
  if (blockIdx.x == 0 && threadIdx.x < HKV) vsmax[threadIdx.x] = 0u;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode3(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
            uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
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
  if (!fn) return PA_ECUDA;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? PA_OK
             : PA_ECUDA;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int pa_prefill_noalloc(int n_q_heads, int n_kv_heads, int n_pool_pages, int max_pages_per_seq,
                                  const void* q, const int8_t* k_pool, const int8_t* v_pool, const float* k_scale,
                                  const float* v_scale, const int32_t* block_table, int q_start, int n_q, int n_ctx,
                                  int n_sink_blk, int n_win_blk, float sm_scale, void* out, void* stream) {
  // argument checks (the same rules as pa_create / pa_prefill)
  if (n_q_heads <= 0 || n_kv_heads <= 0 || n_kv_heads > 8 || n_q_heads % n_kv_heads) return PA_EINVAL;
  const int G = n_q_heads / n_kv_heads;
  if (G > kRows || kRows % G) return PA_EINVAL;
  if (n_pool_pages <= 0 || max_pages_per_seq <= 0 || n_sink_blk < 0) return PA_EINVAL;
  if (n_q < 1 || q_start < 0 || (long long)n_ctx < (long long)q_start + n_q ||
      (long long)n_ctx > (long long)max_pages_per_seq * kPage)
    return PA_EINVAL;
  // positions stay far from int overflow in the unit and tile arithmetic
  if ((long long)q_start + n_q > (1LL << 30) || (long long)n_ctx > (1LL << 30)) return PA_EINVAL;
  if (!q || !k_pool || !v_pool || !k_scale || !v_scale || !block_table || !out) return PA_EINVAL;
  if (!aligned_to(q, 16) || !aligned_to(k_pool, 16) || !aligned_to(v_pool, 16) || !aligned_to(out, 16) ||
      !aligned_to(k_scale, 4) || !aligned_to(v_scale, 4) || !aligned_to(block_table, 4))
    return PA_EINVAL;
  if (!(sm_scale == sm_scale) || sm_scale < 0.f) return PA_EINVAL;
  const int TQ = kRows / G;      // tokens per CTA
  const int UT = kUnitRows / G;  // tokens per unit (a CTA pair)

  SeqGeom sg{};
  sg.q_off = 0;
  sg.q_start = q_start;
  sg.n_q = n_q;
  sg.n_ctx = n_ctx;
  sg.tok_off = 0;
  sg.bt_row = 0;
  seq_geom_fill(sg, n_sink_blk, n_win_blk);
  const long long n_rows = (long long)sg.n_blocks * kPage;
  const int t_first = (q_start / UT) * UT;
  const int n_t0 = (q_start + n_q - 1 - t_first) / UT + 1;
  // size limits of the static scratch: a clear error, never an overflow
  const long long row_bytes = (long long)n_kv_heads * (2 * kHeadDim * 2LL + 2 * sizeof(float));  // bf16 K + fp16 V^T, two scales
  const long long cap_rows = ((long long)PA_NOALLOC_SCRATCH_BYTES - (long long)kWidenedOffset) / row_bytes / 64 * 64;
  if (n_rows > cap_rows || (long long)n_t0 * n_kv_heads > kMaxUnits || n_t0 > kMaxT0) return PA_ENOSCRATCH;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ECUDA;
  DeviceSetup ds;
  int rc = device_setup(dev, &ds);
  if (rc) return rc;
  if (!ds.sm103) return PA_EARCH;
  unsigned char* base = static_cast<unsigned char*>(ds.addr);

  // carve the scratch
  const int cap = (int)cap_rows;  // row stride of the widened buffers
  int* err = reinterpret_cast<int*>(base);
  unsigned int* vsmax = reinterpret_cast<unsigned int*>(base + 256);
  SeqGeom* seq_dev = reinterpret_cast<SeqGeom*>(base + 512);
  Unit* units = reinterpret_cast<Unit*>(base + kHeaderBytes);
  unsigned char* w = base + kWidenedOffset;
  __nv_bfloat16* kw = reinterpret_cast<__nv_bfloat16*>(w);
  w += (size_t)n_kv_heads * cap * kHeadDim * 2;
  __half* vt = reinterpret_cast<__half*>(w);
  w += (size_t)n_kv_heads * cap * kHeadDim * 2;
  float* ks = reinterpret_cast<float*>(w);
  w += (size_t)n_kv_heads * cap * sizeof(float);
  float* vs = reinterpret_cast<float*>(w);

  AttnMaps m;
  if ((rc = encode3(&m.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kw, kHeadDim, n_rows, n_kv_heads, kHeadDim * 2,
                    (uint64_t)cap * kHeadDim * 2, 64, kTileKeys / 2, 1)))
    return rc;
  if ((rc = encode3(&m.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, vt, n_rows, kHeadDim, n_kv_heads, (uint64_t)cap * 2,
                    (uint64_t)cap * kHeadDim * 2, kChunkKeys, kHeadDim / 2, 1)))
    return rc;
  if ((rc = encode3(&m.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, kHeadDim, n_q_heads, n_q, kHeadDim * 2,
                    (uint64_t)n_q_heads * kHeadDim * 2, 64, G, TQ)))
    return rc;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  noalloc_plan_kernel<<<(n_t0 + kPlanThreads - 1) / kPlanThreads, kPlanThreads, 0, st>>>(
      sg, n_sink_blk, n_win_blk, n_kv_heads, UT, n_t0, t_first, seq_dev, units, vsmax, err);
  if (cudaGetLastError() != cudaSuccess) return PA_ECUDA;

  WidenParams wp{};
  wp.k_pool = k_pool;
  wp.v_pool = v_pool;
  wp.k_scale = k_scale;
  wp.v_scale = v_scale;
  wp.block_table = block_table;
  wp.bt_stride = max_pages_per_seq;
  wp.n_pool = n_pool_pages;
  wp.HKV = n_kv_heads;
  wp.seqs = seq_dev;
  wp.n_seq = 1;
  wp.n_stored_blocks = sg.n_blocks;
  wp.n_tok_cap = cap;
  wp.kw = kw;
  wp.vt = vt;
  wp.ks = ks;
  wp.vs = vs;
  wp.vsmax = vsmax;
  wp.err = err;
  wp.k_mult = sm_scale * 1.4426950408889634f;  // the softmax's sm_scale * log2(e), folded into the K scales
  if (launch_widen(wp, st) != cudaSuccess) return PA_ECUDA;

  AttnParams a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.total_q = n_q;
  a.seqs = seq_dev;
  a.units = units;
  a.n_units = n_t0 * n_kv_heads;
  a.ks = ks;
  a.vs = vs;
  a.vsmax = vsmax;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.gate = nullptr;
  a.HQ = n_q_heads;
  a.HKV = n_kv_heads;
  a.G = G;
  a.TQ = TQ;
  a.n_tok_cap = cap;
  a.S = n_sink_blk;
  a.W = n_win_blk;
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  a.q_mode = PA_Q_BF16;
  a.p_mode = PA_P_F16;
  a.err = err;
  a.wait_ns = 2000ull * 1000000ull;
  a.q_ready = nullptr;
  a.debug_stall = 0;
  if (launch_attention(a, m, ds.n_sm, st) != cudaSuccess) return PA_ECUDA;

  // synchronous: report this call's device-side status, read on `stream`
  // behind the kernels (no other stream is waited for)
  int e = 0;
  if (cudaMemcpyAsync(&e, err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return PA_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ECUDA;
  if (e & DEV_ERR_TIMEOUT) return PA_ETIMEOUT;
  if (e & DEV_ERR_BAD_PAGE) return PA_EBADPAGE;
  return e ? PA_ECUDA : PA_OK;
}

// Debug export (tests): the work list the last call on the current device
// built, read back from the scratch array on `stream`.
int pa_debug_noalloc_units(int n_units, int32_t* units_out, void* stream) {
  if (n_units <= 0 || n_units > kMaxUnits || !units_out) return PA_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ECUDA;
  DeviceSetup ds;
  const int rc = device_setup(dev, &ds);
  if (rc) return rc;
  if (!ds.sm103) return PA_EARCH;
  static_assert(sizeof(Unit) == 4 * sizeof(int32_t), "a unit is four int32");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(units_out, static_cast<unsigned char*>(ds.addr) + kHeaderBytes, (size_t)n_units * sizeof(Unit),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return PA_ECUDA;
  return PA_OK;
}
