// moe_route.cu -- expert-major dispatch, row gather and deterministic combine.
//
// Dispatch ("Dist-MoE" note, "What it is selling": route on GPU; nvfp4moe README,
// "Grouped GEMM": contiguous expert-major rows and m_indptr of length E+1 with
// empty experts valid; "MoE layer"/"Training": deterministic permutation and
// combine metadata, padded offsets) is a stable counting sort of the T*k routed
// elements by expert, in three launches:
//   1. k_route_count    per 1024-element chunk: validate ids, per-expert histogram
//   2. k_route_scan     one CTA: per-expert scan over chunks, warp-shuffle prefix
//                       scan over experts into m_indptr / off_pad, m-tile table,
//                       padding rows, expert order for weight-gradient scheduling
//   3. k_route_scatter  per chunk: stable rank of each element among equal experts
//                       (warp match + per-warp counts), write row_of / token_of /
//                       score_of
// Padded row layout: expert e owns rows [off_pad[e], off_pad[e+1]), its segment
// rounded up to the 128-row GEMM tile so no tile straddles two experts.
//
// Gather and combine are HBM-bound row copies with 16-byte vector accesses, one
// warp per row (gather) or per token (combine); the combine sums each token's k
// rows in fixed j order in fp32 ("MoE layer": deterministic combine).

#include <climits>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kChunk = 1024;   // routed elements per dispatch CTA
constexpr int kMaxE = 256;

__device__ __forceinline__ bool element_valid(const int32_t* ids, int f, int k, int E, int* e_out) {
  const int t = f / k;
  const int j = f - t * k;
  const int e = ids[f];
  *e_out = e;
  if (e < 0 || e >= E) return false;
  for (int jj = 0; jj < j; ++jj)
    if (ids[t * k + jj] == e) return false;
  return true;
}

__global__ void __launch_bounds__(kChunk) k_route_count(RouteArgs a) {
  pdl_wait();   // the previous kernel of the stream has completed
  __shared__ int hist[kMaxE];
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int R = a.T * a.k;
  const int f = blockIdx.x * kChunk + threadIdx.x;
  if (f < R) {
    int e;
    if (element_valid(a.ids, f, a.k, a.E, &e)) {
      atomicAdd(&hist[e], 1);
    } else {
      atomicMin(&a.err->first_bad, f);
      atomicCAS(&a.err->code, 0, 4 /*MOE_ERR_BAD_IDS*/);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) a.blockcounts[blockIdx.x * a.E + i] = hist[i];
  pdl_trigger();
}

// Inclusive warp scan with shuffles.
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__global__ void __launch_bounds__(kMaxE) k_route_scan(RouteArgs a) {
  pdl_wait();   // the previous kernel of the stream has completed
  __shared__ int cnt[kMaxE];
  __shared__ int warp_tot[2][kMaxE / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  // 1. per expert: exclusive scan of the chunk histograms -> chunk bases.  The
  // counts are read 16 at a time before any base is written, so the loads of a
  // batch are in flight together instead of one memory round trip per chunk.
  int c = 0;
  if (tid < E) {
    constexpr int kB = 16;
    for (int b0 = 0; b0 < a.nblk; b0 += kB) {
      int v[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u)
        v[u] = b0 + u < a.nblk ? a.blockcounts[(b0 + u) * E + tid] : 0;
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        if (b0 + u < a.nblk) a.blockcounts[(b0 + u) * E + tid] = c;
        c += v[u];
      }
    }
    a.counts[tid] = c;
  }
  cnt[tid] = tid < E ? c : 0;
  // 2. warp-level prefix scans over experts: exact counts and padded counts
  const int p = tid < E ? (c + a.BM - 1) / a.BM * a.BM : 0;
  const int ic = warp_incl_scan(tid < E ? c : 0, lane);
  const int ip = warp_incl_scan(p, lane);
  if (lane == 31) {
    warp_tot[0][warp] = ic;
    warp_tot[1][warp] = ip;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x / 32;
    int t0 = lane < nw ? warp_tot[0][lane] : 0;
    int t1 = lane < nw ? warp_tot[1][lane] : 0;
    const int s0 = warp_incl_scan(t0, lane), s1 = warp_incl_scan(t1, lane);
    if (lane < nw) {
      warp_tot[0][lane] = s0 - t0;   // exclusive warp bases
      warp_tot[1][lane] = s1 - t1;
    }
  }
  __syncthreads();
  const int ec = warp_tot[0][warp] + ic - (tid < E ? c : 0);
  const int ep = warp_tot[1][warp] + ip - p;
  if (tid < E) {
    a.m_indptr[tid] = ec;
    a.off_pad[tid] = ep;
    if (tid == E - 1) {
      a.m_indptr[E] = ec + c;
      a.off_pad[E] = ep + p;
      *a.num_mtiles = (ep + p) / kBM;          // 128-row GEMM m tiles
    }
  }
  __syncthreads();
  if (tid < E) {
    // m tiles of this expert, and its padding rows
    for (int r = ep; r < ep + p; r += kBM) a.tile_expert[r / kBM] = tid;
    for (int r = ep + c; r < ep + p; ++r) {
      a.token_of[r] = -1;
      a.score_of[r] = 0.f;
    }
    // order for weight-gradient tiles: experts with more rows first (ties: lower id)
    int pos = 0;
    for (int e2 = 0; e2 < E; ++e2) {
      const int c2 = cnt[e2];
      pos += (c2 > c) || (c2 == c && e2 < tid);
    }
    a.expert_order[pos] = tid;
  }
  if (tid == 0) {
    int ne = 0;
    for (int e2 = 0; e2 < E; ++e2) ne += cnt[e2] > 0;
    *a.num_nonempty = ne;
  }
  if (a.pair_list) {
    // CTA-pair tile lists: expert e's m tiles [f, f+mt) go two at a time to the
    // pair kernel (pair_list), an odd last one to the one-CTA kernel (left_list)
    const int mt = p / kBM;
    const int np = mt >> 1, nl = mt & 1;
    const int ipp = warp_incl_scan(np, lane), ipl = warp_incl_scan(nl, lane);
    __syncthreads();                       // warp_tot reused
    if (lane == 31) {
      warp_tot[0][warp] = ipp;
      warp_tot[1][warp] = ipl;
    }
    __syncthreads();
    if (warp == 0) {
      const int nw = blockDim.x / 32;
      int t0 = lane < nw ? warp_tot[0][lane] : 0;
      int t1 = lane < nw ? warp_tot[1][lane] : 0;
      const int s0 = warp_incl_scan(t0, lane), s1 = warp_incl_scan(t1, lane);
      if (lane < nw) {
        warp_tot[0][lane] = s0 - t0;
        warp_tot[1][lane] = s1 - t1;
      }
    }
    __syncthreads();
    const int bp = warp_tot[0][warp] + ipp - np;   // exclusive bases
    const int bl = warp_tot[1][warp] + ipl - nl;
    if (tid < E) {
      const int f = ep / kBM;
      for (int j = 0; j < np; ++j) a.pair_list[bp + j] = f + 2 * j;
      if (nl) a.left_list[bl] = f + mt - 1;
      if (tid == E - 1) {
        *a.num_pairs = bp + np;
        *a.num_left = bl + nl;
      }
    }
  }
  pdl_trigger();
}

__global__ void __launch_bounds__(kChunk) k_route_scatter(RouteArgs a) {
  pdl_wait();   // the previous kernel of the stream has completed
  __shared__ int wcnt[kChunk / 32][kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  for (int i = tid; i < (kChunk / 32) * E; i += kChunk) wcnt[i / E][i % E] = 0;
  __syncthreads();
  const int R = a.T * a.k;
  const int f = blockIdx.x * kChunk + tid;
  int e = -1;
  bool valid = false;
  if (f < R) valid = element_valid(a.ids, f, a.k, E, &e);
  const int key = valid ? e : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (valid && lane == __ffs(peers) - 1) wcnt[warp][e] = __popc(peers);
  __syncthreads();
  if (valid) {
    int base = 0;
    for (int w = 0; w < warp; ++w) base += wcnt[w][e];
    const int pos = a.off_pad[e] + a.blockcounts[blockIdx.x * E + e] + base + rank_w;
    a.row_of[f] = pos;
    a.token_of[pos] = f / a.k;
    a.score_of[pos] = a.scores[f];
  } else if (f < R) {
    a.row_of[f] = -1;
  }
  pdl_trigger();
}

// ---------------------------------------------------------------------------

// One warp per pair of rows: both rows' 16-byte vectors are loaded before any is
// stored (2 x 8 loads in flight per lane), and the next pair's token ids are
// fetched before this pair's data.
__global__ void __launch_bounds__(256) k_gather_rows(const uint4* __restrict__ src,
                                                     const int32_t* __restrict__ token_of,
                                                     const int32_t* __restrict__ nrows_p, int nvec,
                                                     uint4* __restrict__ dst) {
  pdl_wait();   // the previous kernel of the stream has completed
  constexpr int U = 8;                     // vectors per lane per row and pass
  const int nrows = *nrows_p;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  int r = 2 * gw;
  int t0 = r < nrows ? token_of[r] : -1;
  int t1 = r + 1 < nrows ? token_of[r + 1] : -1;
  for (; r < nrows; r += 2 * nw) {
    const int rn = r + 2 * nw;
    const int n0 = rn < nrows ? token_of[rn] : -1;
    const int n1 = rn + 1 < nrows ? token_of[rn + 1] : -1;
    const bool has1 = r + 1 < nrows;
    const uint4* s0 = src + (long long)(t0 < 0 ? 0 : t0) * nvec;
    const uint4* s1 = src + (long long)(t1 < 0 ? 0 : t1) * nvec;
    uint4* o0 = dst + (long long)r * nvec;
    uint4* o1 = o0 + nvec;
    for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
      uint4 b0[U], b1[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        b0[u] = (t0 >= 0 && v < nvec) ? s0[v] : make_uint4(0, 0, 0, 0);
        b1[u] = (t1 >= 0 && v < nvec) ? s1[v] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < nvec) {          // streaming stores: the rows are written once here
          __stcs(o0 + v, b0[u]);
          if (has1) __stcs(o1 + v, b1[u]);
        }
      }
    }
    t0 = n0;
    t1 = n1;
  }
  pdl_trigger();
}

__device__ __forceinline__ void acc8(float* acc, const uint4 v) {
  acc[0] += __uint_as_float(v.x << 16); acc[1] += __uint_as_float(v.x & 0xFFFF0000u);
  acc[2] += __uint_as_float(v.y << 16); acc[3] += __uint_as_float(v.y & 0xFFFF0000u);
  acc[4] += __uint_as_float(v.z << 16); acc[5] += __uint_as_float(v.z & 0xFFFF0000u);
  acc[6] += __uint_as_float(v.w << 16); acc[7] += __uint_as_float(v.w & 0xFFFF0000u);
}

// One warp per token.  For small k (<= 8, the common case) every contribution's
// 16-byte vectors are loaded before any is added, so k*U loads per lane are in
// flight; the fp32 sums still run in j order.
template <int KMAX>
__global__ void __launch_bounds__(256) k_combine(const uint4* __restrict__ rows,
                                                 const int32_t* __restrict__ row_of, int T, int k,
                                                 int nvec, uint4* __restrict__ y,
                                                 const float* __restrict__ pdscore, int n_pd,
                                                 float* __restrict__ dscores) {
  pdl_wait();   // the previous kernel of the stream has completed
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  // 16-byte vectors per lane per pass: with k = 8 one (8 loads in flight per lane
  // keep the registers, and so the resident warps, low; measured faster than 2)
  constexpr int U = KMAX <= 4 ? 4 : 1;
  for (int t = gw; t < T; t += nw) {
    int rj[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) rj[j] = j < k ? row_of[t * k + j] : -1;
    for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
      uint4 buf[KMAX][U];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        const uint4* src = rows + (long long)(rj[j] < 0 ? 0 : rj[j]) * nvec;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + lane + 32 * u;
          // streaming loads: each expert row is read once, here
          buf[j][u] = (rj[j] >= 0 && v < nvec) ? __ldcs(src + v) : make_uint4(0, 0, 0, 0);
        }
      }
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (rj[j] >= 0)
#pragma unroll
          for (int u = 0; u < U; ++u) acc8(acc[u], buf[j][u]);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < nvec) {
          uint4 o;
          o.x = pack_bf2(acc[u][0], acc[u][1]);
          o.y = pack_bf2(acc[u][2], acc[u][3]);
          o.z = pack_bf2(acc[u][4], acc[u][5]);
          o.w = pack_bf2(acc[u][6], acc[u][7]);
          y[(long long)t * nvec + v] = o;
        }
      }
    }
    if (dscores) {
      for (int j = lane; j < k; j += 32) {
        const int r = row_of[t * k + j];
        float s = 0.f;
        if (r >= 0)
          for (int nt = 0; nt < n_pd; ++nt) s += pdscore[(long long)r * n_pd + nt];
        dscores[t * k + j] = s;
      }
    }
  }
  pdl_trigger();
}

// Any k: contributions are loaded and added one j at a time (fixed j order).
__global__ void __launch_bounds__(256) k_combine_any(const uint4* __restrict__ rows,
                                                     const int32_t* __restrict__ row_of, int T,
                                                     int k, int nvec, uint4* __restrict__ y,
                                                     const float* __restrict__ pdscore, int n_pd,
                                                     float* __restrict__ dscores) {
  pdl_wait();   // the previous kernel of the stream has completed
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  constexpr int U = 4;
  for (int t = gw; t < T; t += nw) {
    for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
      for (int j = 0; j < k; ++j) {
        const int r = row_of[t * k + j];
        if (r < 0) continue;
        const uint4* src = rows + (long long)r * nvec;
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + lane + 32 * u;
          buf[u] = v < nvec ? __ldcs(src + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) acc8(acc[u], buf[u]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < nvec) {
          uint4 o;
          o.x = pack_bf2(acc[u][0], acc[u][1]);
          o.y = pack_bf2(acc[u][2], acc[u][3]);
          o.z = pack_bf2(acc[u][4], acc[u][5]);
          o.w = pack_bf2(acc[u][6], acc[u][7]);
          y[(long long)t * nvec + v] = o;
        }
      }
    }
    if (dscores) {
      for (int j = lane; j < k; j += 32) {
        const int r = row_of[t * k + j];
        float s = 0.f;
        if (r >= 0)
          for (int nt = 0; nt < n_pd; ++nt) s += pdscore[(long long)r * n_pd + nt];
        dscores[t * k + j] = s;
      }
    }
  }
  pdl_trigger();
}

// Caller-provided expert-major layout (moe_forward_routed): check m_indptr and
// off_pad, list the m tiles that hold routed rows, and copy row_of with entries
// outside the laid-out rows replaced by -1.  Every CTA checks the layout (E+1
// entries); CTA 0 writes the tile list, all CTAs copy row_of.  An inconsistent
// layout lists no tiles, drops every row_of entry and records
// MOE_ERR_INVALID_ARG with the first offending expert as detail; an out-of-range
// row_of entry (checked only on a consistent layout) records detail
// E + 1 + its flat index.
__global__ void __launch_bounds__(kMaxE) k_routed_prepare(RoutedArgs a) {
  pdl_wait();   // the previous kernel of the stream has completed
  __shared__ int bad_s;
  __shared__ int warp_tot[kMaxE / 32];
  const int tid = threadIdx.x;
  const int E = a.E;
  if (tid == 0) bad_s = INT_MAX;
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) {
    const int o = a.off_pad[e];
    bool ok = o >= 0 && (o & (kRoutedGranule - 1)) == 0 && (long long)o <= a.rows;
    if (e == 0) ok = ok && o == 0 && a.m_indptr[0] == 0;
    if (e < E) {
      const int m = a.m_indptr[e + 1] - a.m_indptr[e];
      ok = ok && m >= 0 && a.off_pad[e + 1] - o >= m;
    }
    if (!ok) atomicMin(&bad_s, e);
  }
  __syncthreads();
  const bool valid = bad_s == INT_MAX;
  const int nrows = valid ? a.off_pad[E] : 0;
  if (blockIdx.x == 0) {
    if (!valid && tid == 0) {
      atomicMin(&a.err->first_bad, bad_s);
      atomicCAS(&a.err->code, 0, 1 /*MOE_ERR_INVALID_ARG*/);
    }
    // m tiles per expert: those holding its routed rows (ceil(m_e / 128))
    const int lane = tid & 31, warp = tid >> 5;
    const int nt = (valid && tid < E) ? (a.m_indptr[tid + 1] - a.m_indptr[tid] + kRoutedGranule - 1) /
                                            kRoutedGranule
                                      : 0;
    const int inc = warp_incl_scan(nt, lane);
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      const int nw = blockDim.x / 32;
      const int t0 = lane < nw ? warp_tot[lane] : 0;
      const int s0 = warp_incl_scan(t0, lane);
      if (lane < nw) warp_tot[lane] = s0 - t0;
    }
    __syncthreads();
    const int base = warp_tot[warp] + inc - nt;
    if (tid < E) {
      const int mt0 = a.off_pad[tid] / kRoutedGranule;
      for (int i = 0; i < nt; ++i) {
        a.mtile_list[base + i] = mt0 + i;
        a.tile_expert[mt0 + i] = tid;
      }
    }
    if (tid == blockDim.x - 1) *a.list_count = base + nt;   // the last thread's end = the total
  }
  const int Tk = a.Tk;
  for (int f = blockIdx.x * blockDim.x + tid; f < Tk; f += gridDim.x * blockDim.x) {
    const int r = a.row_of_in[f];
    const bool in = r >= 0 && r < nrows;
    a.row_of_out[f] = in ? r : -1;
    if (valid && r >= nrows) {
      atomicMin(&a.err->first_bad, E + 1 + f);
      atomicCAS(&a.err->code, 0, 1 /*MOE_ERR_INVALID_ARG*/);
    }
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream) {
  cudaError_t e = launch_pdl(k_route_count, dim3(a.nblk), dim3(kChunk), 0, stream, a);
  if (e == cudaSuccess) e = launch_pdl(k_route_scan, dim3(1), dim3(kMaxE), 0, stream, a);
  if (e == cudaSuccess) e = launch_pdl(k_route_scatter, dim3(a.nblk), dim3(kChunk), 0, stream, a);
  return e;
}

cudaError_t launch_routed_prepare(const RoutedArgs& a, int grid, cudaStream_t stream) {
  if (a.E < 1 || a.E > kMaxE) return cudaErrorInvalidValue;
  return launch_pdl(k_routed_prepare, dim3(grid), dim3(kMaxE), 0, stream, a);
}

cudaError_t launch_gather_rows(const void* src, const int32_t* token_of, const int32_t* nrows,
                               int d, void* dst, int grid, cudaStream_t stream) {
  return launch_pdl(k_gather_rows, dim3(grid), dim3(256), 0, stream,
                    static_cast<const uint4*>(src), token_of, nrows, d / 8,
                    static_cast<uint4*>(dst));
}

cudaError_t launch_combine(const void* rows, const int32_t* row_of, int T, int k, int d, void* y,
                           const float* pdscore, int n_pd, float* dscores, int grid,
                           cudaStream_t stream) {
  const uint4* r4 = static_cast<const uint4*>(rows);
  uint4* y4 = static_cast<uint4*>(y);
  if (k <= 4)
    return launch_pdl(k_combine<4>, dim3(grid), dim3(256), 0, stream, r4, row_of, T, k, d / 8,
                      y4, pdscore, n_pd, dscores);
  else if (k <= 8)
    return launch_pdl(k_combine<8>, dim3(grid), dim3(256), 0, stream, r4, row_of, T, k, d / 8,
                      y4, pdscore, n_pd, dscores);
  else
    return launch_pdl(k_combine_any, dim3(grid), dim3(256), 0, stream, r4, row_of, T, k, d / 8,
                      y4, pdscore, n_pd, dscores);
}

}  // namespace moe
