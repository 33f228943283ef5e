// C ABI of the selective-scan forward (declared in include/ssm_scan.h): argument
// checks, chunk planning, tensor maps, the stream-ordered workspace pool and
// kernel dispatch.
#include "ssm_scan.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "bwd_kernel.h"
#include "kernel_table.cuh"
#include "scan_internal.h"

namespace {

using ssm::ScanParams;

// ----------------------------------------------------------------- options

std::atomic<int64_t> g_opt_chunks{0};
std::atomic<int64_t> g_opt_min_chunk_len{64};
std::atomic<int64_t> g_opt_lanes{0};
std::atomic<int64_t> g_opt_lane_threads{32768};
std::atomic<int64_t> g_opt_ctas_per_sm{3};
std::atomic<int64_t> g_opt_pow_path{1};
std::atomic<int64_t> g_opt_tma{1};
std::atomic<int64_t> g_opt_inject_stall{0};  // tests: 1 + tile index the producer withholds
std::atomic<int64_t> g_opt_one_launch{0};    // chunked calls in one launch (decoupled lookback)
std::atomic<int64_t> g_opt_hold_chunk{0};    // tests: 1 + chunk index that never publishes
std::atomic<uint64_t> g_launches{0};

__device__ int g_status;  // raised by a kernel: kStatusTimeout, or any other nonzero value

// ------------------------------------------------------------- profiling

struct ProfRec {
  int kind;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
constexpr int kKinds = 6;
const char* const kKindName[kKinds] = {"ssm_chunk_aggregate", "ssm_scan_output", "ssm_step",
                                      "ssm_bwd_reverse_aggregate", "ssm_bwd_main", "ssm_scan_one_launch"};

// ------------------------------------------------------- per-device pools

std::mutex g_pool_mu;
std::vector<cudaMemPool_t> g_pools;  // index = device ordinal; nullptr = not created

cudaError_t get_pool(int dev, cudaMemPool_t* out) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  if ((int)g_pools.size() <= dev) g_pools.resize(dev + 1, nullptr);
  if (!g_pools[dev]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof props);
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    cudaError_t e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;  // keep freed blocks for reuse: no allocation in steady state
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
    g_pools[dev] = pool;
  }
  *out = g_pools[dev];
  return cudaSuccess;
}

// ---------------------------------------------------------------- planning

struct Plan {
  int S = 0, G = 0;      // states per lane, lanes per channel
  bool tma = false;      // TMA-pipelined tiles (else the generic global-memory path)
  int nchunks = 1;
  int64_t chunk_len = 0;
  ssm::KernelInfo out_k, agg_k, one_k;
};

// var 0: the scan as stated; 1: exact ZOH input term; 2: block prologue (conv + silu).
ssm::KernelInfo lookup(int io, bool lti, int S, int G, int pass, int var) {
  if (var == 2) {
    if (lti) return ssm::KernelInfo();
    return io == SSM_F32 ? ssm::lookup_f32_tv_conv(S, G, pass) : ssm::lookup_bf16_tv_conv(S, G, pass);
  }
  if (var == 1) {
    if (io == SSM_F32) return lti ? ssm::lookup_f32_lti_zoh(S, G, pass) : ssm::lookup_f32_tv_zoh(S, G, pass);
    return lti ? ssm::lookup_bf16_lti_zoh(S, G, pass) : ssm::lookup_bf16_tv_zoh(S, G, pass);
  }
  if (io == SSM_F32) return lti ? ssm::lookup_f32_lti(S, G, pass) : ssm::lookup_f32_tv(S, G, pass);
  return lti ? ssm::lookup_bf16_lti(S, G, pass) : ssm::lookup_bf16_tv(S, G, pass);
}

// Padded state count: the next power of two >= max(N, 2).
int padded_states(int64_t N) {
  int ns = 2;
  while (ns < N) ns *= 2;
  return ns;
}

// A tensor map needs 16-byte row pitches: the channel row of x / delta / z and, for
// time-varying B / C, the state row, which must also fill the kernel's padded row
// (N a power of two).
bool tma_ok(const ssm_dims& d) {
  const int64_t esz = d.io_dtype == SSM_BF16 ? 2 : 4;
  if ((d.dim * esz) % 16) return false;
  if (d.bc_layout == SSM_BC_TIME_VARYING &&
      ((d.dstate * esz) % 16 || padded_states(d.dstate) != d.dstate))
    return false;
  if (d.seqlen >= (1ll << 31) || d.dim >= (1ll << 31) || d.batch >= (1ll << 31)) return false;
  return true;
}

// Sets the kernel's shared-memory limit once (it may exceed the 48 KB default).
bool prepare(const ssm::KernelInfo& k) {
  static std::mutex mu;
  static std::vector<const void*> done;
  std::lock_guard<std::mutex> lk(mu);
  for (auto f : done)
    if (f == (const void*)k.fn) return true;
  if (cudaFuncSetAttribute((const void*)k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem) !=
      cudaSuccess)
    return false;
  done.push_back((const void*)k.fn);
  return true;
}

// Resident CTAs per SM of a kernel (cached).
int occupancy(const ssm::KernelInfo& k) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> cache;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (auto& e : cache)
      if (e.first == (const void*)k.fn) return e.second;
  }
  int occ = 0;
  if (!prepare(k) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, (const void*)k.fn, k.nt, k.smem) != cudaSuccess ||
      occ < 1)
    occ = 1;
  std::lock_guard<std::mutex> lk(mu);
  cache.push_back({(const void*)k.fn, occ});
  return occ;
}

// Lanes per channel: the fewest (least per-state overhead) that give at least
// `lane_threads` threads over the batch rows and channels; one otherwise (the
// sequence is then chunked).
// Workspace of the two-kernel chunk carry with k chunks: end states and step sums of
// chunks 0 .. k-2, a copy of the initial state and of the prologue's input history.
size_t chunk_ws_bytes(const ssm_dims& d, int64_t k, bool conv) {
  if (k <= 1) return 0;
  const size_t nH = (size_t)(k - 1) * d.batch * d.dim * d.dstate;
  const size_t nS = (size_t)(k - 1) * d.batch * d.dim;
  const size_t nh0 = d.state_in ? (size_t)d.batch * d.dim * d.dstate : 0;
  const size_t ncs = (conv && d.state_in) ? (size_t)d.batch * d.dim * 3 : 0;
  return (nH + nS + nh0 + ncs) * sizeof(float);
}

// Workspace of the one-launch carry with k chunks: the publication flags and the ticket
// counter (cleared before every launch), the step sums and end states of chunks
// 1 .. k-2 (slots indexed by chunk), the first chunk's true end state and a copy of the
// initial state.
struct OneLaunchWs {
  size_t flag_bytes = 0, off_S = 0, off_H = 0, off_P = 0, off_h0 = 0, bytes = 0;
};

constexpr int kConsumerWarps = 4;  // per CTA of the tiled kernel: one publication flag each

OneLaunchWs one_launch_ws(const ssm_dims& d, int64_t k, int ch) {
  OneLaunchWs w;
  if (k <= 1) return w;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  const int nwb = (int)((d.dim + ch - 1) / ch) * kConsumerWarps;
  const size_t nflags = (size_t)(k - 1) * d.batch * nwb + 1;
  const size_t nS = (size_t)(k - 1) * d.batch * d.dim;
  const size_t st = (size_t)d.batch * d.dim * d.dstate;
  w.flag_bytes = up(nflags * 4);
  w.off_S = w.flag_bytes;
  w.off_H = w.off_S + up(nS * 4);
  w.off_P = w.off_H + up(nS * d.dstate * 4);
  w.off_h0 = w.off_P + up(st * 4);
  w.bytes = w.off_h0 + (d.state_in ? up(st * 4) : 0);
  return w;
}

// The workspace a call with k chunks needs, in the carry mode the options select.
size_t call_ws_bytes(const ssm_dims& d, int64_t k, bool conv, int ch) {
  return g_opt_one_launch.load() ? one_launch_ws(d, k, ch).bytes : chunk_ws_bytes(d, k, conv);
}

// Chunks along the sequence only when that leaves fewer than `ctas_per_sm` CTAs per
// SM: every chunk but the last is then scanned twice (aggregate, output), so the
// chunk count is the largest that still fits ctas_per_sm CTAs on every SM (one
// wave, evenly spread).
bool make_plan(const ssm_dims& d, int sms, bool conv, Plan* pl, size_t max_ws_bytes) {
  const int ns = padded_states(d.dstate);
  const bool lti = d.bc_layout == SSM_BC_PER_CHANNEL;
  std::vector<int> cand;
  for (int G = 1; G <= 4; G *= 2) {
    const int S = ns / G;
    if (S >= 2 && S <= 16 && lookup(d.io_dtype, lti, S, G, 1, conv ? 2 : 0).fn) cand.push_back(G);
  }
  if (cand.empty()) return false;
  const int64_t forced = g_opt_lanes.load();
  int G = 0;
  if (forced > 0) {
    for (int c : cand)
      if (c == forced) G = c;
    if (!G) return false;
  } else if (d.io_dtype == SSM_F32) {
    // fp32 inputs carry decays as Abar - 1 (two more FMA-pipe operations per state):
    // one lane per channel amortises the per-step work best; chunks fill the GPU
    G = cand.front();
  } else {
    // the fewest lanes that reach lane_threads; if even the most cannot, the sequence
    // must be chunked anyway, and one lane per channel (least per-state work) is best
    G = cand.front();
    for (int c : cand)
      if (d.batch * d.dim * c >= g_opt_lane_threads.load()) {
        G = c;
        break;
      }
  }
  pl->G = G;
  pl->S = ns / G;
  const int var = conv ? 2 : d.bbar_mode;
  pl->out_k = lookup(d.io_dtype, lti, pl->S, G, 1, var);
  pl->agg_k = lookup(d.io_dtype, lti, pl->S, G, 0, var);
  pl->one_k = lookup(d.io_dtype, lti, pl->S, G, 2, var);
  pl->tma = g_opt_tma.load() && tma_ok(d);
  int64_t k = g_opt_chunks.load();
  if (k <= 0) {
    const int64_t ctas = d.batch * ((d.dim + pl->out_k.ch - 1) / pl->out_k.ch);
    const int64_t per_sm = std::max<int64_t>(
        1, std::min<int64_t>(g_opt_ctas_per_sm.load(), occupancy(pl->out_k)));
    const int64_t want = (int64_t)sms * per_sm;
    k = ctas >= want ? 1 : std::max<int64_t>(1, want / ctas);
    const int64_t min_len = std::max<int64_t>(ssm::kChunkAlign, g_opt_min_chunk_len.load());
    k = std::min<int64_t>(k, std::max<int64_t>(1, d.seqlen / min_len));
  }
  k = std::max<int64_t>(1, std::min<int64_t>(k, (d.seqlen + ssm::kChunkAlign - 1) / ssm::kChunkAlign));
  k = std::min<int64_t>(k, 65535);
  // chunk length: a multiple of kChunkAlign steps, so tiles never straddle chunks
  auto split = [&](int64_t kk) {
    int64_t len = (d.seqlen + kk - 1) / kk;
    len = ((len + ssm::kChunkAlign - 1) / ssm::kChunkAlign) * ssm::kChunkAlign;
    pl->chunk_len = std::max<int64_t>(len, ssm::kChunkAlign);
    pl->nchunks = (int)((d.seqlen + pl->chunk_len - 1) / pl->chunk_len);
  };
  split(k);
  if (max_ws_bytes && g_opt_chunks.load() <= 0) {
    // a fixed scratch: fewer automatic chunks until the workspace fits
    while (pl->nchunks > 1 && call_ws_bytes(d, pl->nchunks, conv, pl->out_k.ch) > max_ws_bytes)
      split(pl->nchunks - 1);
  }
  return true;
}

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a row-major (batch, rows, inner) tensor with a box of (inner_box, rows_box, 1).
bool encode3d(CUtensorMap* m, const void* base, int esz, int64_t inner, int64_t rows, int64_t batch,
              int inner_box, int rows_box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)batch};
  const cuuint64_t strides[2] = {(cuuint64_t)(inner * esz), (cuuint64_t)(inner * rows * esz)};
  const cuuint32_t box[3] = {(cuuint32_t)inner_box, (cuuint32_t)rows_box, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch(const ssm::KernelInfo& kn, int kind, dim3 grid, const ssm::TmaMaps& maps, const ScanParams& p,
           cudaStream_t stream) {
  if (!kn.fn || !prepare(kn)) return SSM_ERR_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  bool prof;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    prof = g_prof_on;
  }
  if (prof) {
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return SSM_ERR_CUDA;
    if (cudaEventRecord(e0, stream) != cudaSuccess) return SSM_ERR_CUDA;
  }
  kn.fn<<<grid, kn.nt, kn.smem, stream>>>(maps, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return SSM_ERR_CUDA;
  g_launches.fetch_add(1);
  if (prof) {
    if (cudaEventRecord(e1, stream) != cudaSuccess) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back({kind, e0, e1});
  }
  return SSM_OK;
}

// Launch of a backward-pass kernel (one warp per CTA), with the same profiling hook.
int launch_bwd(ssm::BwdFn fn, int kind, dim3 grid, const ssm::BwdParams& p, cudaStream_t stream) {
  if (!fn) return SSM_ERR_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  bool prof;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    prof = g_prof_on;
  }
  if (prof) {
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return SSM_ERR_CUDA;
    if (cudaEventRecord(e0, stream) != cudaSuccess) return SSM_ERR_CUDA;
  }
  fn<<<grid, 32, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
  g_launches.fetch_add(1);
  if (prof) {
    if (cudaEventRecord(e1, stream) != cudaSuccess) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back({kind, e0, e1});
  }
  return SSM_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" {

const char* ssm_status_string(int code) {
  switch (code) {
    case SSM_OK: return "ok";
    case SSM_ERR_NULL: return "a required pointer is NULL";
    case SSM_ERR_DIMS: return "invalid sizes or flags";
    case SSM_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case SSM_ERR_UNSUPPORTED: return "mode not implemented in this build";
    case SSM_ERR_CUDA: return "CUDA runtime error";
    case SSM_ERR_OVERLAP: return "an output overlaps another tensor";
    case SSM_ERR_NOMEM: return "workspace allocation failed";
    case SSM_ERR_DEVICE: return "a kernel reported an internal inconsistency";
    case SSM_ERR_TIMEOUT: return "a kernel gave up waiting for its copies";
    case SSM_ERR_SCRATCH: return "the call needs more scratch than the fixed no-allocation buffer holds";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace ssm_internal {

void count_launch() { g_launches.fetch_add(1); }

cudaError_t workspace_pool(int dev, cudaMemPool_t* out) { return get_pool(dev, out); }

int* status_word() {
  int* status = nullptr;
  if (cudaGetSymbolAddress((void**)&status, g_status) != cudaSuccess) return nullptr;
  return status;
}

// The whole call.  scratch == nullptr: the chunk-carry workspace comes from the
// library's stream-ordered pool.  Otherwise it is carved from `scratch`
// (scratch_bytes long, device memory the caller keeps), nothing is allocated, and a
// call whose workspace does not fit returns SSM_ERR_SCRATCH before launching.
int scan_forward(const void* x, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* delta_bias, void* out,
                 float* final_state, const ssm_dims* dims, cudaStream_t stream, void* scratch,
                 size_t scratch_bytes, const ConvPrologue* conv) {
  if (!dims) return SSM_ERR_NULL;
  const ssm_dims d = *dims;
  if (d.batch <= 0 || d.dim <= 0 || d.dstate <= 0 || d.dstate > 64 || d.seqlen < 0)
    return SSM_ERR_DIMS;
  if ((d.io_dtype != SSM_F32 && d.io_dtype != SSM_BF16) ||
      (d.bc_layout != SSM_BC_TIME_VARYING && d.bc_layout != SSM_BC_PER_CHANNEL) ||
      (d.delta_softplus != 0 && d.delta_softplus != 1) || (d.state_in != 0 && d.state_in != 1) ||
      (d.bbar_mode != 0 && d.bbar_mode != 1) || d.reserved != 0)
    return SSM_ERR_DIMS;
  if (d.state_in && !final_state) return SSM_ERR_DIMS;
  if (d.seqlen > 0 && (!x || !delta || !A || !B || !C || !out)) return SSM_ERR_NULL;
  const void* ptrs[] = {x, delta, A, B, C, D, z, delta_bias, out, final_state};
  for (const void* q : ptrs)
    if (q && ((uintptr_t)q & 15u)) return SSM_ERR_ALIGN;
  if (conv) {
    if (!conv->w) return SSM_ERR_NULL;
    const void* cptrs[] = {conv->w, conv->b, conv->state};
    for (const void* q : cptrs)
      if (q && ((uintptr_t)q & 15u)) return SSM_ERR_ALIGN;
    // the prologue form: time-varying B and C and the fused scan's input term
    if (d.bc_layout != SSM_BC_TIME_VARYING || d.bbar_mode != 0) return SSM_ERR_UNSUPPORTED;
  }
  float* const cstate = conv ? conv->state : nullptr;
  const float* const chist = (conv && d.state_in) ? conv->state : nullptr;

  const size_t esz = d.io_dtype == SSM_BF16 ? 2 : 4;
  const size_t act = (size_t)d.batch * d.seqlen * d.dim * esz;
  const bool lti = d.bc_layout == SSM_BC_PER_CHANNEL;
  const size_t bc = lti ? (size_t)d.dim * d.dstate * 4 : (size_t)d.batch * d.seqlen * d.dstate * esz;
  const size_t st = (size_t)d.batch * d.dim * d.dstate * 4;
  struct { const void* p; size_t n; } ins[] = {
      {x, act}, {delta, act}, {A, (size_t)d.dim * d.dstate * 4}, {B, bc}, {C, bc},
      {D, (size_t)d.dim * 4}, {z, act}, {delta_bias, (size_t)d.dim * 4}};
  for (auto& in : ins) {
    if (overlaps(out, act, in.p, in.n)) return SSM_ERR_OVERLAP;
    if (overlaps(final_state, st, in.p, in.n)) return SSM_ERR_OVERLAP;
  }
  if (overlaps(final_state, st, out, act)) return SSM_ERR_OVERLAP;
  const size_t cst = (size_t)d.batch * d.dim * 3 * 4;
  if (cstate) {
    for (auto& in : ins)
      if (overlaps(cstate, cst, in.p, in.n)) return SSM_ERR_OVERLAP;
    if (overlaps(cstate, cst, out, act) || overlaps(cstate, cst, final_state, st) ||
        overlaps(cstate, cst, conv->w, (size_t)d.dim * 16) || overlaps(cstate, cst, conv->b, (size_t)d.dim * 4))
      return SSM_ERR_OVERLAP;
  }

  if (d.seqlen == 0) {
    if (final_state && !d.state_in &&
        cudaMemsetAsync(final_state, 0, st, stream) != cudaSuccess)
      return SSM_ERR_CUDA;
    if (cstate && !d.state_in && cudaMemsetAsync(cstate, 0, cst, stream) != cudaSuccess)
      return SSM_ERR_CUDA;
    return SSM_OK;
  }

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;

  if (d.seqlen == 1) {
    // recurrent step: one pass over the state, no tiles, no chunks, no workspace
    int ns = 4;
    while (ns < d.dstate) ns *= 2;
    const int G = ns / 4;
    const ssm::KernelInfo k = ssm::lookup_step(d.io_dtype == SSM_BF16, lti, G, conv != nullptr);
    if (!k.fn) return SSM_ERR_UNSUPPORTED;
    ScanParams p;
    std::memset(&p, 0, sizeof p);
    if (conv) {
      p.conv_w = conv->w; p.conv_b = conv->b; p.conv_hist_in = chist; p.conv_state_out = cstate;
    }
    p.x = x; p.delta = delta; p.z = z; p.out = out; p.A = A; p.B = B; p.C = C;
    p.Dskip = D; p.bias = delta_bias; p.final_state = final_state;
    p.h_init = d.state_in ? final_state : nullptr;
    p.batch = d.batch; p.seqlen = 1; p.dim = d.dim; p.dstate = (int)d.dstate;
    p.nchunks = 1; p.chunk_len = 1;
    p.delta_softplus = d.delta_softplus;
    p.bbar_mode = d.bbar_mode;
    ssm::TmaMaps maps;
    std::memset(&maps, 0, sizeof maps);
    const int64_t threads = d.batch * d.dim * G;
    if ((threads + k.nt - 1) / k.nt > INT32_MAX) return SSM_ERR_DIMS;
    return launch(k, 2, dim3((unsigned)((threads + k.nt - 1) / k.nt)), maps, p, stream);
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SSM_ERR_CUDA;
  if (d.batch > 65535) return SSM_ERR_DIMS;
  Plan pl;
  if (!make_plan(d, sms, conv != nullptr, &pl, scratch ? scratch_bytes : 0)) return SSM_ERR_UNSUPPORTED;

  ScanParams p;
  std::memset(&p, 0, sizeof p);
  p.x = x; p.delta = delta; p.z = z; p.out = out; p.A = A; p.B = B; p.C = C;
  p.Dskip = D; p.bias = delta_bias; p.final_state = final_state;
  p.h_init = d.state_in ? final_state : nullptr;
  p.batch = d.batch; p.seqlen = d.seqlen; p.dim = d.dim; p.dstate = (int)d.dstate;
  p.nchunks = pl.nchunks; p.chunk_len = pl.chunk_len;
  p.delta_softplus = d.delta_softplus;
  p.pow_path = (int)g_opt_pow_path.load();
  p.use_tma = pl.tma ? 1 : 0;
  p.bbar_mode = d.bbar_mode;
  p.stall_tile = (int)g_opt_inject_stall.load() - 1;
  if (conv) {
    p.conv_w = conv->w; p.conv_b = conv->b; p.conv_hist_in = chist; p.conv_state_out = cstate;
  }
  int* status = nullptr;
  if (cudaGetSymbolAddress((void**)&status, g_status) != cudaSuccess) return SSM_ERR_CUDA;
  p.status = status;

  const int ch = pl.out_k.ch, T = pl.out_k.t;
  const unsigned gx = (unsigned)((d.dim + ch - 1) / ch);

  ssm::TmaMaps maps;
  std::memset(&maps, 0, sizeof maps);
  if (pl.tma) {
    const int eb = (int)esz;
    bool okm = encode3d(&maps.x, x, eb, d.dim, d.seqlen, d.batch, ch, T) &&
               encode3d(&maps.delta, delta, eb, d.dim, d.seqlen, d.batch, ch, T);
    if (okm && z) okm = encode3d(&maps.z, z, eb, d.dim, d.seqlen, d.batch, ch, T);
    // the output pass writes out in tiles of the x box
    if (okm) okm = encode3d(&maps.out, out, eb, d.dim, d.seqlen, d.batch, ch, T);
    if (okm && !lti)
      okm = encode3d(&maps.B, B, eb, d.dstate, d.seqlen, d.batch, (int)d.dstate, T) &&
            encode3d(&maps.C, C, eb, d.dstate, d.seqlen, d.batch, (int)d.dstate, T);
    if (!okm) return SSM_ERR_CUDA;
  }

  if (pl.nchunks > 1 && g_opt_one_launch.load()) {
    // the whole call in one launch: aggregates published with flags, decoupled lookback
    const OneLaunchWs w = one_launch_ws(d, pl.nchunks, ch);
    const int64_t nblocks = (int64_t)pl.nchunks * d.batch * gx;
    if (nblocks > INT32_MAX) return SSM_ERR_DIMS;
    void* ws1 = nullptr;
    unsigned char* base = nullptr;
    if (scratch) {
      if (w.bytes > scratch_bytes) return SSM_ERR_SCRATCH;
      base = static_cast<unsigned char*>(scratch);
    } else {
      cudaMemPool_t pool;
      if (get_pool(dev, &pool) != cudaSuccess) return SSM_ERR_CUDA;
      if (cudaMallocFromPoolAsync(&ws1, w.bytes, pool, stream) != cudaSuccess) return SSM_ERR_NOMEM;
      base = static_cast<unsigned char*>(ws1);
    }
    p.ncb = (int)gx;
    p.nwb = (int)gx * kConsumerWarps;
    p.hold_chunk = (int)g_opt_hold_chunk.load() - 1;
    p.flags = reinterpret_cast<unsigned*>(base);
    p.ticket = p.flags + (size_t)(pl.nchunks - 1) * d.batch * p.nwb;
    p.ws_S = reinterpret_cast<float*>(base + w.off_S);
    p.ws_H = reinterpret_cast<float*>(base + w.off_H);
    p.ws_P = reinterpret_cast<float*>(base + w.off_P);
    p.ws_h0 = d.state_in ? reinterpret_cast<float*>(base + w.off_h0) : nullptr;
    int rc = cudaMemsetAsync(base, 0, w.flag_bytes, stream) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    if (rc == SSM_OK) rc = launch(pl.one_k, 5, dim3((unsigned)nblocks), maps, p, stream);
    if (ws1 && cudaFreeAsync(ws1, stream) != cudaSuccess && rc == SSM_OK) rc = SSM_ERR_CUDA;
    return rc;
  }

  void* ws = nullptr;
  if (pl.nchunks > 1) {
    const size_t nH = (size_t)(pl.nchunks - 1) * d.batch * d.dim * d.dstate;
    const size_t nS = (size_t)(pl.nchunks - 1) * d.batch * d.dim;
    const size_t nh0 = d.state_in ? (size_t)d.batch * d.dim * d.dstate : 0;
    // the prologue's input history, copied by the aggregate pass: the output pass
    // writes the new history over the same buffer
    const size_t ncs = chist ? (size_t)d.batch * d.dim * 3 : 0;
    const size_t bytes = chunk_ws_bytes(d, pl.nchunks, conv != nullptr);
    if (scratch) {
      if (bytes > scratch_bytes) return SSM_ERR_SCRATCH;
      p.ws_H = static_cast<float*>(scratch);
    } else {
      cudaMemPool_t pool;
      if (get_pool(dev, &pool) != cudaSuccess) return SSM_ERR_CUDA;
      if (cudaMallocFromPoolAsync(&ws, bytes, pool, stream) != cudaSuccess) return SSM_ERR_NOMEM;
      p.ws_H = static_cast<float*>(ws);
    }
    p.ws_S = p.ws_H + nH;
    p.ws_h0 = nh0 ? p.ws_S + nS : nullptr;
    p.ws_cs = ncs ? p.ws_S + nS + nh0 : nullptr;
    int rc = launch(pl.agg_k, 0, dim3(gx, (unsigned)(pl.nchunks - 1), (unsigned)d.batch), maps, p, stream);
    if (rc != SSM_OK) {
      if (ws) cudaFreeAsync(ws, stream);
      return rc;
    }
  }
  int rc = launch(pl.out_k, 1, dim3(gx, (unsigned)pl.nchunks, (unsigned)d.batch), maps, p, stream);
  if (ws && cudaFreeAsync(ws, stream) != cudaSuccess && rc == SSM_OK) rc = SSM_ERR_CUDA;
  return rc;
}

// Gradients of one selective-scan call (bbar_mode 0, time-varying B and C, N <= 16).
int scan_backward(const void* x, const void* delta, const float* A, const void* B, const void* C,
                  const float* D, const void* z, const float* delta_bias, const float* h_init,
                  const void* dout, const float* dfinal, void* dx, void* ddelta, float* dA, float* dB,
                  float* dC, float* dD, void* dz, float* ddelta_bias, float* dh_init,
                  const ssm_dims* dims, cudaStream_t stream) {
  if (!dims) return SSM_ERR_NULL;
  const ssm_dims d = *dims;
  if (d.batch <= 0 || d.dim <= 0 || d.dstate <= 0 || d.dstate > 64 || d.seqlen < 0)
    return SSM_ERR_DIMS;
  if ((d.io_dtype != SSM_F32 && d.io_dtype != SSM_BF16) ||
      (d.bc_layout != SSM_BC_TIME_VARYING && d.bc_layout != SSM_BC_PER_CHANNEL) ||
      (d.delta_softplus != 0 && d.delta_softplus != 1) || (d.state_in != 0 && d.state_in != 1) ||
      (d.bbar_mode != 0 && d.bbar_mode != 1) || d.reserved != 0)
    return SSM_ERR_DIMS;
  if (d.bc_layout != SSM_BC_TIME_VARYING || d.bbar_mode != 0 || d.dstate > 16) return SSM_ERR_UNSUPPORTED;
  if (!A || !dA) return SSM_ERR_NULL;
  if (d.seqlen > 0 && (!x || !delta || !B || !C || !dout || !dx || !ddelta || !dB || !dC))
    return SSM_ERR_NULL;
  if (z && !dz) return SSM_ERR_NULL;
  const void* ptrs[] = {x, delta, A, B, C, D, z, delta_bias, h_init, dout, dfinal, dx, ddelta,
                        dA, dB, dC, dD, dz, ddelta_bias, dh_init};
  for (const void* q : ptrs)
    if (q && ((uintptr_t)q & 15u)) return SSM_ERR_ALIGN;
  const size_t esz = d.io_dtype == SSM_BF16 ? 2 : 4;
  const size_t act = (size_t)d.batch * d.seqlen * d.dim * esz;
  const size_t bcn = (size_t)d.batch * d.seqlen * d.dstate;
  const size_t st = (size_t)d.batch * d.dim * d.dstate * 4;
  struct { const void* p; size_t n; } ins[] = {
      {x, act}, {delta, act}, {A, (size_t)d.dim * d.dstate * 4}, {B, bcn * esz}, {C, bcn * esz},
      {D, (size_t)d.dim * 4}, {z, act}, {delta_bias, (size_t)d.dim * 4}, {h_init, st}, {dout, act},
      {dfinal, st}};
  struct { const void* p; size_t n; } outs[] = {
      {dx, act}, {ddelta, act}, {dA, (size_t)d.dim * d.dstate * 4}, {dB, bcn * 4}, {dC, bcn * 4},
      {dD, (size_t)d.dim * 4}, {dz, act}, {ddelta_bias, (size_t)d.dim * 4}, {dh_init, st}};
  for (auto& o : outs) {
    for (auto& in : ins)
      if (overlaps(o.p, o.n, in.p, in.n)) return SSM_ERR_OVERLAP;
    for (auto& o2 : outs)
      if (&o2 != &o && overlaps(o.p, o.n, o2.p, o2.n)) return SSM_ERR_OVERLAP;
  }

  // the shared gradients are sums: start from zero
  if (cudaMemsetAsync(dA, 0, (size_t)d.dim * d.dstate * 4, stream) != cudaSuccess) return SSM_ERR_CUDA;
  if (dD && cudaMemsetAsync(dD, 0, (size_t)d.dim * 4, stream) != cudaSuccess) return SSM_ERR_CUDA;
  if (ddelta_bias && cudaMemsetAsync(ddelta_bias, 0, (size_t)d.dim * 4, stream) != cudaSuccess)
    return SSM_ERR_CUDA;
  if (d.seqlen == 0) {
    // the final state is the initial one
    if (dh_init) {
      cudaError_t e = dfinal ? cudaMemcpyAsync(dh_init, dfinal, st, cudaMemcpyDeviceToDevice, stream)
                             : cudaMemsetAsync(dh_init, 0, st, stream);
      if (e != cudaSuccess) return SSM_ERR_CUDA;
    }
    return SSM_OK;
  }
  if (cudaMemsetAsync(dB, 0, bcn * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(dC, 0, bcn * 4, stream) != cudaSuccess)
    return SSM_ERR_CUDA;

  const int S = padded_states(d.dstate);
  const ssm::BwdKernels bk = ssm::lookup_bwd(d.io_dtype == SSM_BF16, S);
  const ssm::KernelInfo agg = lookup(d.io_dtype, false, S, 1, 0, 0);
  if (!bk.main || !agg.fn) return SSM_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SSM_ERR_CUDA;
  if (d.batch > 65535) return SSM_ERR_DIMS;

  // chunks: one warp per 32 channels and chunk; as many chunks as fill every SM with
  // the main kernel's resident CTAs in one wave (chunks of at least min_chunk_len steps)
  const unsigned gx = (unsigned)((d.dim + 31) / 32);
  int64_t k = g_opt_chunks.load();
  if (k <= 0) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, (const void*)bk.main, 32, 0) != cudaSuccess ||
        occ < 1)
      occ = 8;
    const int64_t warps = d.batch * gx, want = (int64_t)sms * occ;
    k = warps >= want ? 1 : std::max<int64_t>(1, want / warps);
    k = std::min<int64_t>(k, std::max<int64_t>(1, d.seqlen / std::max<int64_t>(ssm::kChunkAlign,
                                                                                 g_opt_min_chunk_len.load())));
  }
  k = std::max<int64_t>(1, std::min<int64_t>(k, (d.seqlen + ssm::kChunkAlign - 1) / ssm::kChunkAlign));
  k = std::min<int64_t>(k, 65535);
  int64_t len = (d.seqlen + k - 1) / k;
  len = ((len + ssm::kChunkAlign - 1) / ssm::kChunkAlign) * ssm::kChunkAlign;
  const int nchunks = (int)((d.seqlen + len - 1) / len);

  // the reverse aggregate pass (a light kernel, 32 resident CTAs per SM) runs rsub
  // sub-chunks per chunk (at most 4, a power of two, so that sub-chunks stay multiples
  // of 8 steps) to come near 32 warps per SM
  int rsub = 1;
  if (nchunks > 1) {
    const int64_t warps = (int64_t)(nchunks - 1) * d.batch * gx;
    while (rsub < 4 && warps * rsub * 2 <= (int64_t)sms * 32) rsub *= 2;
  }
  const size_t nH = (size_t)(nchunks - 1) * d.batch * d.dim * d.dstate;
  const size_t nS = (size_t)(nchunks - 1) * d.batch * d.dim;
  const size_t nM = nH * rsub, nS2 = nS * rsub;
  const size_t nck = (size_t)((d.seqlen + bk.seg - 1) / bk.seg) * d.batch * d.dim * S;
  const size_t bytes = (nH + nS + nM + nS2 + nck) * sizeof(float);
  cudaMemPool_t pool;
  if (get_pool(dev, &pool) != cudaSuccess) return SSM_ERR_CUDA;
  void* ws = nullptr;
  if (cudaMallocFromPoolAsync(&ws, bytes, pool, stream) != cudaSuccess) return SSM_ERR_NOMEM;
  float* const w0 = static_cast<float*>(ws);

  ssm::BwdParams bp;
  std::memset(&bp, 0, sizeof bp);
  bp.x = x; bp.delta = delta; bp.z = z; bp.A = A; bp.B = B; bp.C = C; bp.Dskip = D;
  bp.bias = delta_bias; bp.h_init = h_init; bp.dout = dout; bp.dfinal = dfinal;
  bp.dx = dx; bp.ddelta = ddelta; bp.dz = dz; bp.dA = dA; bp.dB = dB; bp.dC = dC; bp.dD = dD;
  bp.dbias = ddelta_bias; bp.dh_init = dh_init;
  bp.ws_H = w0; bp.ws_S = w0 + nH; bp.ws_M = w0 + nH + nS; bp.ws_S2 = w0 + nH + nS + nM;
  bp.ws_ck = w0 + nH + nS + nM + nS2;
  bp.batch = d.batch; bp.seqlen = d.seqlen; bp.dim = d.dim; bp.dstate = (int)d.dstate;
  bp.nchunks = nchunks; bp.chunk_len = len; bp.delta_softplus = d.delta_softplus;
  bp.rsub = rsub; bp.rsub_len = len / rsub;

  int rc = SSM_OK;
  if (nchunks > 1) {
    // forward chunk aggregates: the tiled forward kernel's aggregate pass
    ScanParams p;
    std::memset(&p, 0, sizeof p);
    p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.bias = delta_bias; p.h_init = h_init;
    p.ws_H = w0; p.ws_S = w0 + nH;
    p.batch = d.batch; p.seqlen = d.seqlen; p.dim = d.dim; p.dstate = (int)d.dstate;
    p.nchunks = nchunks; p.chunk_len = len; p.delta_softplus = d.delta_softplus;
    p.pow_path = (int)g_opt_pow_path.load();
    p.stall_tile = -1;
    int* status = nullptr;
    if (cudaGetSymbolAddress((void**)&status, g_status) != cudaSuccess) rc = SSM_ERR_CUDA;
    p.status = status;
    ssm::TmaMaps maps;
    std::memset(&maps, 0, sizeof maps);
    const bool tma = g_opt_tma.load() && tma_ok(d);
    p.use_tma = tma ? 1 : 0;
    if (rc == SSM_OK && tma) {
      const int eb = (int)esz;
      if (!encode3d(&maps.x, x, eb, d.dim, d.seqlen, d.batch, agg.ch, agg.t) ||
          !encode3d(&maps.delta, delta, eb, d.dim, d.seqlen, d.batch, agg.ch, agg.t) ||
          !encode3d(&maps.B, B, eb, d.dstate, d.seqlen, d.batch, (int)d.dstate, agg.t))
        rc = SSM_ERR_CUDA;
    }
    if (rc == SSM_OK)
      rc = launch(agg, 0, dim3((unsigned)((d.dim + agg.ch - 1) / agg.ch), (unsigned)(nchunks - 1),
                               (unsigned)d.batch), maps, p, stream);
    if (rc == SSM_OK)
      rc = launch_bwd(bk.reverse_aggregate, 3, dim3(gx, (unsigned)((nchunks - 1) * rsub), (unsigned)d.batch),
                      bp, stream);
  }
  if (rc == SSM_OK) rc = launch_bwd(bk.main, 4, dim3(gx, (unsigned)nchunks, (unsigned)d.batch), bp, stream);
  if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == SSM_OK) rc = SSM_ERR_CUDA;
  return rc;
}

}  // namespace ssm_internal

extern "C" {

int ssm_selective_scan_bwd(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z, const float* delta_bias,
                           const float* h_init, const void* dout, const float* dfinal_state,
                           void* dx, void* ddelta, float* dA, float* dB, float* dC, float* dD,
                           void* dz, float* ddelta_bias, float* dh_init, const ssm_dims* dims,
                           cudaStream_t stream) {
  return ssm_internal::scan_backward(x, delta, A, B, C, D, z, delta_bias, h_init, dout, dfinal_state,
                                     dx, ddelta, dA, dB, dC, dD, dz, ddelta_bias, dh_init, dims, stream);
}


int ssm_selective_scan_fwd(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const float* delta_bias, void* out, float* final_state,
                           const ssm_dims* dims, cudaStream_t stream) {
  return ssm_internal::scan_forward(x, delta, A, B, C, D, z, delta_bias, out, final_state, dims, stream,
                                    nullptr, 0, nullptr);
}

int ssm_conv_selective_scan_fwd(const void* x, const float* conv_w, const float* conv_b,
                                float* conv_state, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z,
                                const float* delta_bias, void* out, float* final_state,
                                const ssm_dims* dims, cudaStream_t stream) {
  const ssm_internal::ConvPrologue cp{conv_w, conv_b, conv_state};
  return ssm_internal::scan_forward(x, delta, A, B, C, D, z, delta_bias, out, final_state, dims, stream,
                                    nullptr, 0, &cp);
}

int ssm_check_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SSM_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return SSM_ERR_CUDA;
  if (v == 0) return SSM_OK;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof zero) != cudaSuccess) return SSM_ERR_CUDA;
  return v == ssm::kStatusTimeout ? SSM_ERR_TIMEOUT : SSM_ERR_DEVICE;
}

int ssm_release_workspace(void) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return SSM_ERR_CUDA;
  int rc = SSM_OK;
  for (int dev = 0; dev < (int)g_pools.size(); ++dev) {
    if (!g_pools[dev]) continue;
    if (cudaSetDevice(dev) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemPoolTrimTo(g_pools[dev], 0) != cudaSuccess)
      rc = SSM_ERR_CUDA;
  }
  cudaSetDevice(cur);
  return rc;
}

uint64_t ssm_kernel_launches(void) { return g_launches.load(); }

int64_t ssm_workspace_reserved_bytes(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_pool_mu);
  if (dev >= (int)g_pools.size() || !g_pools[dev]) return 0;
  cuuint64_t v = 0;
  if (cudaMemPoolGetAttribute(g_pools[dev], cudaMemPoolAttrReservedMemCurrent, &v) != cudaSuccess)
    return SSM_ERR_CUDA;
  return (int64_t)v;
}

int ssm_set_option(const char* name, int64_t value) {
  if (!name || value < 0) return SSM_ERR_DIMS;
  if (!std::strcmp(name, "chunks")) g_opt_chunks = value;
  else if (!std::strcmp(name, "min_chunk_len")) g_opt_min_chunk_len = value;
  else if (!std::strcmp(name, "lanes")) g_opt_lanes = value;
  else if (!std::strcmp(name, "lane_threads")) g_opt_lane_threads = value;
  else if (!std::strcmp(name, "ctas_per_sm")) g_opt_ctas_per_sm = value;
  else if (!std::strcmp(name, "pow_path")) g_opt_pow_path = value ? 1 : 0;
  else if (!std::strcmp(name, "tma")) g_opt_tma = value ? 1 : 0;
  else if (!std::strcmp(name, "inject_stall")) g_opt_inject_stall = std::min<int64_t>(value, INT32_MAX);
  else if (!std::strcmp(name, "one_launch")) g_opt_one_launch = value ? 1 : 0;
  else if (!std::strcmp(name, "hold_chunk")) g_opt_hold_chunk = std::min<int64_t>(value, INT32_MAX);
  else if (!ssm_internal::set_ssd_option(name, value)) return SSM_ERR_DIMS;
  return SSM_OK;
}

int ssm_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  return SSM_OK;
}

int ssm_profile_read(const char** names, int64_t* launches, double* total_ms, int max) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
  }
  int64_t cnt[kKinds] = {};
  double ms[kKinds] = {};
  int rc = SSM_OK;
  for (auto& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      rc = SSM_ERR_CUDA;
    cnt[r.kind] += 1;
    ms[r.kind] += t;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  if (rc != SSM_OK) return rc;
  int rows = 0;
  for (int k = 0; k < kKinds; ++k) {
    if (!cnt[k]) continue;
    if (rows < max) {
      if (names) names[rows] = kKindName[k];
      if (launches) launches[rows] = cnt[k];
      if (total_ms) total_ms[rows] = ms[k];
    }
    ++rows;
  }
  return rows;
}

}  // extern "C"
