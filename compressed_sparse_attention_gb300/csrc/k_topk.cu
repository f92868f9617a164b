// Top-k selection S_t = TopK_j sigma_t(j) ("Reading Notes of DeepSeek-V4.1-
// Flash", section 3f, C2 step 2), with ties broken toward the lower index and
// the chosen indices written in ascending order, -1 padded (PocketLLM
// "DeepSeek-V4.1-Flash", "The CSA2 attention layers").
//
// Integer work on the scores' bit patterns:
//   1. hist:   a 4096-bin histogram of the top 12 bits of each score's
//              order-preserving key (per query, over all CTAs of the row);
//   2. filter: every CTA finds the bin that holds the k-th largest key and
//              appends (key, index) of every element at or above it to a
//              per-query candidate list;
//   3. select: one CTA per query runs an exact MSD radix select over the
//              candidates' unique 64-bit composite key<<32 | ~index (larger
//              composite = larger score, then lower index), keeps the
//              composites at or above the threshold, and sorts their indices.
#include "launchers.cuh"

namespace csa2 {

constexpr int kHistBins = 4096;
constexpr int kTopkChunk = 4096;   // scores per CTA in hist / filter
constexpr int kSelCap = 8192;      // candidates held in shared memory by select
constexpr int kMaxTopk = 2048;

__device__ __forceinline__ uint32_t hist_bin(uint32_t key) { return key >> 20; }

__global__ void __launch_bounds__(256) topk_hist_kernel(const float* __restrict__ scores, int64_t ld,
                                                        const int32_t* __restrict__ n_vis, int64_t max_vis,
                                                        uint32_t* __restrict__ hist) {
  __shared__ uint32_t h[kHistBins];
  const int q = blockIdx.y;
  const int nv = (int)min((int64_t)n_vis[q], max_vis);
  const int64_t c0 = (int64_t)blockIdx.x * kTopkChunk;
  if (c0 >= nv) return;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const float* row = scores + (int64_t)q * ld;
  for (int i = threadIdx.x; i < kTopkChunk; i += blockDim.x) {
    const int64_t j = c0 + i;
    const bool ok = j < nv;
    const uint32_t bin = ok ? hist_bin(score_key(row[j])) : 0xFFFFFFFFu;
    const uint32_t peers = __match_any_sync(0xffffffffu, bin);
    if (ok && (__ffs(peers) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&h[bin], (uint32_t)__popc(peers));
  }
  __syncthreads();
  uint32_t* gh = hist + (int64_t)q * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (h[i]) atomicAdd(&gh[i], h[i]);
}

// Bin b* such that count(bin > b*) < need <= count(bin >= b*), from the top.
__device__ uint32_t find_threshold_bin(const uint32_t* __restrict__ gh, uint32_t need, uint32_t* scan_s) {
  // 256 threads, 16 bins each, thread 0 owns the 16 highest bins
  const int tid = threadIdx.x;
  uint32_t local[16], sum = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    local[k] = gh[kHistBins - 1 - (16 * tid + k)];
    sum += local[k];
  }
  scan_s[tid] = sum;
  __syncthreads();
  // inclusive scan (Hillis-Steele) over 256 partial sums
  for (int off = 1; off < 256; off <<= 1) {
    const uint32_t v = tid >= off ? scan_s[tid - off] : 0u;
    __syncthreads();
    scan_s[tid] += v;
    __syncthreads();
  }
  const uint32_t incl = scan_s[tid], excl = incl - sum;
  __syncthreads();
  if (excl < need && need <= incl) {
    uint32_t run = excl;
    for (int k = 0; k < 16; ++k) {
      run += local[k];
      if (run >= need) {
        scan_s[256] = (uint32_t)(kHistBins - 1 - (16 * tid + k));
        break;
      }
    }
  }
  __syncthreads();
  return scan_s[256];
}

__global__ void __launch_bounds__(256) topk_filter_kernel(const float* __restrict__ scores, int64_t ld,
                                                          const int32_t* __restrict__ n_vis, int64_t max_vis,
                                                          int k, const uint32_t* __restrict__ hist,
                                                          uint32_t* __restrict__ cnt,
                                                          unsigned long long* __restrict__ cand,
                                                          int64_t cand_ld) {
  __shared__ uint32_t scan_s[257];
  const int q = blockIdx.y;
  const int nv = (int)min((int64_t)n_vis[q], max_vis);
  const int64_t c0 = (int64_t)blockIdx.x * kTopkChunk;
  if (c0 >= nv) return;
  const uint32_t need = (uint32_t)min(k, nv);
  uint32_t bstar = 0;
  if ((uint32_t)nv > need) bstar = find_threshold_bin(hist + (int64_t)q * kHistBins, need, scan_s);
  const float* row = scores + (int64_t)q * ld;
  unsigned long long* out = cand + (int64_t)q * cand_ld;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kTopkChunk; i += blockDim.x) {
    const int64_t j = c0 + i;
    uint32_t key = 0;
    bool take = false;
    if (j < nv) {
      key = score_key(row[j]);
      take = hist_bin(key) >= bstar;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, take);
    if (m) {
      uint32_t base = 0;
      if (lane == 0) base = atomicAdd(&cnt[q], (uint32_t)__popc(m));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (take) {
        const uint32_t slot = base + __popc(m & ((1u << lane) - 1u));
        out[slot] = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)j);
      }
    }
  }
}

// MSD radix select of the need-th largest value among n unique 64-bit values.
template <typename Src>
__device__ unsigned long long radix_select64(Src src, uint32_t n, uint32_t need, uint32_t* hist_s,
                                             unsigned long long* bcast) {
  unsigned long long prefix = 0, mask = 0;
  uint32_t remaining = need;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist_s[i] = 0;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
      const unsigned long long v = src(i);
      if ((v & mask) == prefix) atomicAdd(&hist_s[(v >> shift) & 0xFF], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // suffix sums over 256 digits: lane owns digits 255-8*lane .. 248-8*lane
      uint32_t loc[8], s = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        loc[u] = hist_s[255 - 8 * threadIdx.x - u];
        s += loc[u];
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if ((int)threadIdx.x >= o) incl += v;
      }
      const uint32_t excl = incl - s;
      if (excl < remaining && remaining <= incl) {
        uint32_t run = excl;
        for (int u = 0; u < 8; ++u) {
          if (run + loc[u] >= remaining) {
            bcast[0] = (unsigned long long)(255 - 8 * threadIdx.x - u);
            bcast[1] = (unsigned long long)(remaining - run);
            break;
          }
          run += loc[u];
        }
      }
    }
    __syncthreads();
    const unsigned long long d = bcast[0];
    remaining = (uint32_t)bcast[1];
    prefix |= d << shift;
    mask |= 0xFFull << shift;
    __syncthreads();
  }
  return prefix;
}

__global__ void __launch_bounds__(1024) topk_select_kernel(const int32_t* __restrict__ n_vis, int64_t max_vis, int k,
                                                           const uint32_t* __restrict__ cnt,
                                                           const unsigned long long* __restrict__ cand,
                                                           int64_t cand_ld, int32_t* __restrict__ out_idx) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  unsigned long long* cs = reinterpret_cast<unsigned long long*>(sm_raw);  // [kSelCap]
  uint32_t* sel = reinterpret_cast<uint32_t*>(cs + kSelCap);               // [kMaxTopk]
  __shared__ uint32_t hist_s[256];
  __shared__ unsigned long long bcast[2];
  __shared__ uint32_t n_sel;
  const int q = blockIdx.x;
  const int nv = (int)min((int64_t)n_vis[q], max_vis);
  const uint32_t need = (uint32_t)max(0, min(k, nv));
  uint32_t n = cnt[q];
  const unsigned long long* gc = cand + (int64_t)q * cand_ld;
  if (n > (uint32_t)max(nv, 0)) n = (uint32_t)max(nv, 0);
  const uint32_t take = min(need, n);
  unsigned long long thr = 0;
  const bool in_smem = n <= (uint32_t)kSelCap;
  if (in_smem)
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) cs[i] = gc[i];
  if (threadIdx.x == 0) n_sel = 0;
  __syncthreads();
  if (take > 0 && take < n) {
    if (in_smem) thr = radix_select64([&](uint32_t i) { return cs[i]; }, n, take, hist_s, bcast);
    else thr = radix_select64([&](uint32_t i) { return gc[i]; }, n, take, hist_s, bcast);
  }
  // collect the chosen indices
  for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long v = in_smem ? cs[i] : gc[i];
    if (take > 0 && v >= thr) {
      const uint32_t slot = atomicAdd(&n_sel, 1u);
      if (slot < (uint32_t)kMaxTopk) sel[slot] = 0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull);
    }
  }
  __syncthreads();
  const uint32_t ns = min(n_sel, (uint32_t)kMaxTopk);
  uint32_t pw = 1;
  while (pw < ns) pw <<= 1;
  for (uint32_t i = ns + threadIdx.x; i < pw; i += blockDim.x) sel[i] = 0xFFFFFFFFu;
  __syncthreads();
  // bitonic sort ascending
  for (uint32_t size = 2; size <= pw; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t i = threadIdx.x; i < pw; i += blockDim.x) {
        const uint32_t jx = i ^ stride;
        if (jx > i) {
          const bool up = (i & size) == 0;
          const uint32_t a = sel[i], b = sel[jx];
          if ((a > b) == up) { sel[i] = b; sel[jx] = a; }
        }
      }
      __syncthreads();
    }
  }
  int32_t* o = out_idx + (int64_t)q * k;
  for (int i = threadIdx.x; i < k; i += blockDim.x) o[i] = (uint32_t)i < ns ? (int32_t)sel[i] : -1;
}

size_t topk_workspace_bytes(int n_query, int64_t max_vis) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)n_query * kHistBins * 4) + al((size_t)n_query * 4) +
         al((size_t)n_query * (size_t)(max_vis > 0 ? max_vis : 1) * 8);
}

cudaError_t launch_topk(cudaStream_t st, int n_query, const float* scores, int64_t ld, const int32_t* n_vis,
                        int64_t max_vis, int k, int32_t* out_idx, void* ws, int* n_launch) {
  if (n_query == 0) return cudaSuccess;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  char* p = reinterpret_cast<char*>(ws);
  uint32_t* hist = reinterpret_cast<uint32_t*>(p);
  p += al((size_t)n_query * kHistBins * 4);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(p);
  p += al((size_t)n_query * 4);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(p);
  const int64_t cand_ld = max_vis > 0 ? max_vis : 1;
  cudaError_t e = cudaMemsetAsync(ws, 0, al((size_t)n_query * kHistBins * 4) + al((size_t)n_query * 4), st);
  if (e != cudaSuccess) return e;
  if (max_vis > 0) {
    const dim3 g((unsigned)((max_vis + kTopkChunk - 1) / kTopkChunk), (unsigned)n_query);
    topk_hist_kernel<<<g, 256, 0, st>>>(scores, ld, n_vis, max_vis, hist);
    topk_filter_kernel<<<g, 256, 0, st>>>(scores, ld, n_vis, max_vis, k, hist, cnt, cand, cand_ld);
    *n_launch += 2;
  }
  const size_t smem = (size_t)kSelCap * 8 + (size_t)kMaxTopk * 4;
  e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_select_kernel<<<n_query, 1024, smem, st>>>(n_vis, max_vis, k, cnt, cand, cand_ld, out_idx);
  *n_launch += 1;
  return cudaGetLastError();
}

}  // namespace csa2
