// moe_static.cu -- expert-major dispatch for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they route tokens: code running inside another framework's allocator
// hooks or memory-pool callbacks, a host that has already carved all device
// memory into fixed pools, or a process that may only touch memory it was
// handed.  For them, moe_dispatch_static runs the same three dispatch kernels
// as moe_forward, but keeps the kernels' scratch (per-chunk expert histograms,
// per-expert counts, the m-tile table, the expert order and the device error
// word) in one file-scope __device__ array of fixed size instead of a
// caller-provided workspace.  The caller passes only its inputs and outputs.
//
// Properties of the static scratch:
//   - every GPU that loads this library holds the array (about 280 KB) until the
//     process exits;
//   - its device address is looked up once per device and CUDA context, by the
//     first call made with that device current (cudaGetSymbolAddress).  A call
//     from another context on the same device (a non-primary context, or the
//     primary one re-created after cudaDeviceReset) looks the address up again,
//     in that context, so it is also a first call;
//   - every call on a device shares the one array and it keeps the last call's
//     contents: the error word is cleared at the start of each call, everything
//     else is fully rewritten; calls whose kernels overlap on the GPU (for
//     example from two streams at once) race on it and must not be issued.

#include <climits>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

namespace {

constexpr int kStaticMaxE = 256;
constexpr int kChunk = 1024;
constexpr long long kStaticMaxRouted = MOE_STATIC_MAX_ROUTED;
constexpr int kStaticMaxChunks = (int)((kStaticMaxRouted + kChunk - 1) / kChunk);
constexpr long long kStaticMaxTiles =
    (kStaticMaxRouted + (long long)kStaticMaxE * (moe::kBM - 1)) / moe::kBM;

// int32 words of the static scratch, in order.
constexpr size_t kOffErr = 0;                                    // DevError (4 words)
constexpr size_t kOffCounts = 64;                                // [E]
constexpr size_t kOffNumMt = kOffCounts + kStaticMaxE;           // scalar
constexpr size_t kOffNumNe = kOffNumMt + 64;                     // scalar
constexpr size_t kOffOrder = kOffNumNe + 64;                     // [E]
constexpr size_t kOffTiles = kOffOrder + kStaticMaxE;            // [max tiles]
constexpr size_t kOffChunks = kOffTiles + ((kStaticMaxTiles + 63) / 64) * 64;   // [chunks, E]
constexpr size_t kWords = kOffChunks + (size_t)kStaticMaxChunks * kStaticMaxE;

__device__ __align__(256) int32_t g_dispatch_scratch[kWords];

std::mutex g_mu;
// per device ordinal: the array's address and the context it was looked up in
int32_t* g_scratch_addr[64] = {nullptr};
CUcontext g_scratch_ctx[64] = {nullptr};

// The calling thread's current CUDA context (driver entry point, looked up once).
CUcontext current_context() {
  static const PFN_cuCtxGetCurrent_v4000 fn = []() -> PFN_cuCtxGetCurrent_v4000 {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Launch without launch attributes, returning the launch's own status (a
// <<<>>> launch leaves it to cudaGetLastError, which also reports and clears
// errors the caller left pending).
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kernel)(KArgs...), cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__global__ void k_static_begin(moe::DevError* err) {
  err->code = 0;
  err->first_bad = INT_MAX;
  err->where = 0;
  err->pad = 0;
}

__global__ void k_static_end(const moe::DevError* err, int32_t* status) {
  status[0] = err->code;
  status[1] = err->code == MOE_ERR_BAD_IDS ? err->first_bad : -1;
}

}  // namespace

extern "C" int moe_dispatch_static(const int32_t* ids, const float* scores, int T, int k, int E,
                                   int32_t* m_indptr, int32_t* off_pad, int32_t* row_of,
                                   int32_t* token_of, float* score_of, long long rows_capacity,
                                   int32_t* status, void* stream) {
  if (!ids || !scores || !m_indptr || !off_pad || !row_of || !token_of || !score_of || !status)
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || E < k || E > kStaticMaxE) return MOE_ERR_INVALID_ARG;
  const long long R = (long long)T * k;
  if (R > kStaticMaxRouted) return MOE_ERR_WORKSPACE;        // beyond the static scratch
  const long long need_rows = (R + (long long)E * (moe::kBM - 1)) / moe::kBM * moe::kBM;
  if (rows_capacity < need_rows) return MOE_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  // NULL until the runtime has made a context current on this thread
  CUcontext ctx = current_context();
  int32_t* base;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ctx || !g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
      // set-up: the array's address in the current context (the lookup also
      // initialises the device's primary context when none is current yet)
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
      ctx = current_context();
      if (!ctx) return MOE_ERR_CUDA;
      g_scratch_addr[dev] = static_cast<int32_t*>(p);
      g_scratch_ctx[dev] = ctx;
    }
    base = g_scratch_addr[dev];
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  moe::DevError* err = reinterpret_cast<moe::DevError*>(base + kOffErr);
  moe::RouteArgs ra{};            // every pointer not set below stays NULL
  ra.ids = ids;
  ra.scores = scores;
  ra.T = T;
  ra.k = k;
  ra.E = E;
  ra.BM = moe::kBM;
  ra.nblk = (int)((R + kChunk - 1) / kChunk);
  ra.blockcounts = base + kOffChunks;
  ra.counts = base + kOffCounts;
  ra.m_indptr = m_indptr;
  ra.off_pad = off_pad;
  ra.num_mtiles = base + kOffNumMt;
  ra.tile_expert = base + kOffTiles;
  ra.expert_order = base + kOffOrder;
  ra.num_nonempty = base + kOffNumNe;
  ra.row_of = row_of;
  ra.token_of = token_of;
  ra.score_of = score_of;
  ra.err = err;
  if (launch_plain(k_static_begin, st, err) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_route(ra, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_plain(k_static_end, st, static_cast<const moe::DevError*>(err), status) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
