// Top-k selection S_t = TopK_j sigma_t(j) ("Reading Notes of DeepSeek-V4.1-
// Flash", section 3f, C2 step 2), with ties broken toward the lower index and
// the chosen indices written in ascending order, -1 padded (PocketLLM
// "DeepSeek-V4.1-Flash", "The CSA2 attention layers").
//
// Integer work on the scores' order-preserving bit patterns. Rows of up to
// 16,384 scores take one launch of one CTA per query. Rows of up to 262,144
// scores take one launch of a thread-block cluster per query running an MSD
// radix select over shared memory (described above the kernel below), when
// all the queries' clusters fit on the GPU at once. Longer rows, and more
// queries than that, take three launches through global memory:
//   1. hist:   a 4096-bin histogram of the top 12 bits of each score's key
//              (per query, over all CTAs of the row);
//   2. filter: every CTA finds the bin that holds the k-th largest key and
//              appends (key, index) of every element at or above it to a
//              per-query candidate list;
//   3. select: one CTA per query runs an exact MSD radix select over the
//              candidates' unique 64-bit composite key<<32 | ~index (larger
//              composite = larger score, then lower index), keeps the
//              composites at or above the threshold, and sorts their indices.
#include <cooperative_groups.h>

#include "launchers.cuh"

namespace csa2 {

constexpr int kHistBins = 4096;
constexpr int kTopkChunk = 4096;   // scores per CTA in hist / filter
constexpr int kTopkBatch = 8;      // loads in flight per thread there
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
  const int len = (int)min((int64_t)kTopkChunk, nv - c0);
  for (int b0 = 0; b0 < len; b0 += 256 * kTopkBatch) {
    float v[kTopkBatch];
#pragma unroll
    for (int u = 0; u < kTopkBatch; ++u) {
      const int i = b0 + u * 256 + (int)threadIdx.x;
      v[u] = i < len ? row[c0 + i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kTopkBatch; ++u) {
      // plain shared-memory atomics: aggregating equal bins across the warp
      // first (match) measured slower, even though the bins are few and hot
      if (b0 + u * 256 + (int)threadIdx.x < len) atomicAdd(&h[hist_bin(score_key(v[u]))], 1u);
    }
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
  const int len = (int)min((int64_t)kTopkChunk, nv - c0);
  for (int b0 = 0; b0 < len; b0 += 256 * kTopkBatch) {
    float v[kTopkBatch];
#pragma unroll
    for (int u = 0; u < kTopkBatch; ++u) {
      const int i = b0 + u * 256 + (int)threadIdx.x;
      v[u] = i < len ? row[c0 + i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kTopkBatch; ++u) {
      const int i = b0 + u * 256 + (int)threadIdx.x;
      const uint32_t key = score_key(v[u]);
      const bool take = i < len && hist_bin(key) >= bstar;
      const uint32_t m = __ballot_sync(0xffffffffu, take);
      if (m) {
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&cnt[q], (uint32_t)__popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (take) {
          const uint32_t slot = base + __popc(m & ((1u << lane) - 1u));
          const uint32_t j = (uint32_t)(c0 + i);
          out[slot] = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - j);
        }
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
      if ((v & mask) == prefix) atomicAdd(&hist_s[(uint32_t)((v >> shift) & 0xFF)], 1u);
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
            bcast[2] = (unsigned long long)loc[u];
            break;
          }
          run += loc[u];
        }
      }
    }
    __syncthreads();
    const unsigned long long d = bcast[0];
    remaining = (uint32_t)bcast[1];
    const bool whole_bin = bcast[2] == (unsigned long long)remaining;
    prefix |= d << shift;
    mask |= 0xFFull << shift;
    __syncthreads();
    // every value in the chosen bin is needed: the threshold is the bin's
    // smallest possible value, whatever the lower digits
    if (whole_bin) break;
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
  __shared__ unsigned long long bcast[3];
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
  // ascending order: the chosen indices are distinct, so each one's output
  // slot is the number of chosen indices below it (the reads of sel[j] are
  // shared-memory broadcasts across the warp)
  int32_t* o = out_idx + (int64_t)q * k;
  for (uint32_t i = threadIdx.x; i < ns; i += blockDim.x) {
    const uint32_t v = sel[i];
    uint32_t r = 0;
    for (uint32_t jx = 0; jx < ns; ++jx) r += sel[jx] < v ? 1u : 0u;
    if (r < (uint32_t)k) o[r] = (int32_t)v;
  }
  for (int i = (int)ns + threadIdx.x; i < k; i += blockDim.x) o[i] = -1;
}

// ---------------------------------------------------------------------------
// Pool sharding (one sequence's pool split over shards [lo, hi)): the
// visible count of a shard, the (score, entry) pairs of a shard's local
// selection, and the merge of the shards' pairs into the global top-k. The
// merge keys each pair by the 64-bit composite key << 32 | ~entry, unique per
// entry, so the k largest composites are the k largest scores with ties to
// the lower entry, exactly the unsharded selection on the same scores.
// ---------------------------------------------------------------------------
__global__ void shard_visible_kernel(int n_query, const int32_t* __restrict__ n_vis, int64_t lo, int64_t hi,
                                     int32_t* __restrict__ out) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= n_query) return;
  const int64_t v = (int64_t)n_vis[q] - lo;
  out[q] = (int32_t)max((int64_t)0, min(v, hi - lo));
}

cudaError_t launch_shard_visible(cudaStream_t st, int n_query, const int32_t* n_vis, int64_t lo, int64_t hi,
                                 int32_t* n_vis_shard, int* n_launch) {
  if (n_query == 0) return cudaSuccess;
  shard_visible_kernel<<<(n_query + 255) / 256, 256, 0, st>>>(n_query, n_vis, lo, hi, n_vis_shard);
  *n_launch += 1;
  return cudaGetLastError();
}

__global__ void topk_pairs_kernel(int n_query, const float* __restrict__ scores, int64_t ld,
                                  const int32_t* __restrict__ sel, int k, int64_t base, float* __restrict__ ps,
                                  int32_t* __restrict__ pi) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)n_query * k) return;
  const int64_t q = i / k;
  const int32_t j = sel[i];
  if (j >= 0) {
    ps[i] = scores[q * ld + j];
    pi[i] = (int32_t)(base + j);
  } else {
    ps[i] = -INFINITY;
    pi[i] = -1;
  }
}

cudaError_t launch_topk_pairs(cudaStream_t st, int n_query, const float* scores, int64_t ld, const int32_t* sel, int k,
                              int64_t index_base, float* pair_score, int32_t* pair_idx, int* n_launch) {
  const int64_t n = (int64_t)n_query * k;
  if (n == 0) return cudaSuccess;
  topk_pairs_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(n_query, scores, ld, sel, k, index_base, pair_score,
                                                                pair_idx);
  *n_launch += 1;
  return cudaGetLastError();
}

__device__ __forceinline__ uint32_t block_scan_incl(uint32_t v, uint32_t* warp_s);  // below

// One 1024-thread CTA per query: pair i of the lists (list-major order)
// becomes the composite key(score) << 32 | ~entry in shared-memory slot i (0
// for an empty pair, below every composite), a radix select finds the k-th
// largest composite, and the chosen entries are written ascending, -1
// padded. Thread t holds slots [t c, t c + c): when the chosen entries come
// out ascending in slot order (each list ascending and the lists' entry
// ranges in list order, as shards' and slices' lists are), a block scan of
// the threads' chosen counts places them; otherwise each is ranked against
// the others. Lists are list-major ([list][query][k_in]); with scores !=
// nullptr (the slices of one row, query-major [query][list][k_in]) a pair's
// score is read from the row, scores[q * ld + entry], instead of from ps.
__global__ void __launch_bounds__(1024) topk_merge_kernel(int n_query, int n_lists, int k_in,
                                                          const float* __restrict__ ps,
                                                          const int32_t* __restrict__ pi, int k,
                                                          int32_t* __restrict__ out_idx,
                                                          const float* __restrict__ scores = nullptr,
                                                          int64_t ld = 0) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  unsigned long long* cs = reinterpret_cast<unsigned long long*>(sm_raw);  // [kSelCap]
  uint32_t* sel = reinterpret_cast<uint32_t*>(cs + kSelCap);               // [kMaxTopk]
  __shared__ uint32_t hist_s[256];
  __shared__ unsigned long long bcast[3];
  __shared__ uint32_t warp_s[32];
  const int q = blockIdx.x;
  pdl_wait();  // the lists of the previous kernel (a plain launch returns at once)
  pdl_trigger();
  const uint32_t total = min((uint32_t)(n_lists * k_in), (uint32_t)kSelCap);
  uint32_t n_valid = 0;
  for (uint32_t i = threadIdx.x; i < total; i += blockDim.x) {
    const uint32_t l = i / (uint32_t)k_in, e = i - l * (uint32_t)k_in;
    const int64_t g = scores != nullptr ? ((int64_t)q * n_lists + l) * k_in + e : ((int64_t)l * n_query + q) * k_in + e;
    const int32_t j = pi[g];
    unsigned long long v = 0ull;
    if (j >= 0) {
      const float sc = scores != nullptr ? scores[(int64_t)q * ld + j] : ps[g];
      v = ((unsigned long long)score_key(sc) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)j);
      ++n_valid;
    }
    cs[i] = v;
  }
  n_valid = __reduce_add_sync(0xffffffffu, n_valid);
  if ((threadIdx.x & 31) == 0) warp_s[threadIdx.x >> 5] = n_valid;
  __syncthreads();  // the slots and the warps' counts are complete
  uint32_t nv = 0;
#pragma unroll
  for (int w = 0; w < 32; ++w) nv += warp_s[w];
  const uint32_t take = min((uint32_t)k, nv);
  unsigned long long thr = 1ull;  // every composite is chosen (empty slots are 0)
  if (take > 0 && take < nv) thr = radix_select64([&](uint32_t i) { return cs[i]; }, total, take, hist_s, bcast);
  // this thread's slots and their chosen count; the chosen entries in slot order
  const uint32_t c = (total + blockDim.x - 1) / blockDim.x;
  const uint32_t s0 = min(total, threadIdx.x * c), s1 = min(total, s0 + c);
  uint32_t cnt = 0;
  for (uint32_t i = s0; i < s1; ++i) {
    const unsigned long long v = cs[i];
    if (take > 0 && v >= thr && v != 0ull) ++cnt;
  }
  const uint32_t pos0 = block_scan_incl(cnt, warp_s) - cnt;  // ends synchronised
  {
    uint32_t p = pos0;
    for (uint32_t i = s0; i < s1; ++i) {
      const unsigned long long v = cs[i];
      if (take > 0 && v >= thr && v != 0ull && p < (uint32_t)kMaxTopk) sel[p++] = 0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull);
    }
  }
  __syncthreads();
  const uint32_t ns = min(take, (uint32_t)kMaxTopk);
  bool ok = true;  // strictly ascending in slot order
  for (uint32_t i = threadIdx.x; i + 1 < ns; i += blockDim.x) ok = ok && sel[i] < sel[i + 1];
  const bool ordered = __syncthreads_and(ok) != 0;
  int32_t* o = out_idx + (int64_t)q * k;
  if (ordered) {
    for (uint32_t i = threadIdx.x; i < ns; i += blockDim.x) o[i] = (int32_t)sel[i];
  } else {
    for (uint32_t i = threadIdx.x; i < ns; i += blockDim.x) {
      const uint32_t v = sel[i];
      uint32_t r = 0;
      for (uint32_t jx = 0; jx < ns; ++jx) r += sel[jx] < v ? 1u : 0u;
      if (r < (uint32_t)k) o[r] = (int32_t)v;
    }
  }
  for (int i = (int)ns + threadIdx.x; i < k; i += blockDim.x) o[i] = -1;
}

cudaError_t launch_topk_merge(cudaStream_t st, int n_query, int n_lists, int k_in, const float* pair_score,
                              const int32_t* pair_idx, int k, int32_t* out_idx, int* n_launch) {
  if (n_query == 0) return cudaSuccess;
  if ((int64_t)n_lists * k_in > kSelCap || k > kMaxTopk) return cudaErrorInvalidValue;
  const size_t smem = (size_t)kSelCap * 8 + (size_t)kMaxTopk * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_merge_kernel<<<n_query, 1024, smem, st>>>(n_query, n_lists, k_in, pair_score, pair_idx, k, out_idx);
  *n_launch += 1;
  return cudaGetLastError();
}

namespace cg = cooperative_groups;

// ---------------------------------------------------------------------------
// Single-launch top-k for rows of up to 8 x 32,768 scores: a thread-block
// cluster of C <= 8 CTAs per query (the portable size: a 1,024-thread CTA
// holds a whole SM, and not every GPC has room for a 16-CTA cluster), CTA r
// holding scores [r*S, (r+1)*S) of the row as order-preserving keys in
// shared memory. Element li of a slice sits in thread li % 1024, round li / 1024,
// so a warp's ballot in round u is bit-word u*32 + warp of the slice's
// bitmap and word w covers elements 32w .. 32w+31.
//   1. (the digits start at the key's top bit);
//   2. MSD digit levels of up to 12 bits: each histograms the keys that match
//      the digits chosen so far and picks the digit that holds the k-th
//      largest key; in a cluster in two stages, first among 64 blocks of
//      bins, then among the bins of the chosen block, each summed over the
//      cluster through distributed shared memory (a one-CTA row scans its
//      own bins at once);
//   3. the search ends as soon as the picked bin
//      - holds exactly the keys still needed: the chosen set is every key
//        whose prefix is at or above the picked one; or
//      - (in a cluster) holds at most 256 keys: they are gathered from the
//        whole cluster and each is ranked against the others by (key
//        descending, index ascending), which takes ties lowest index first; or
//      - is a full 32-bit key T held by more keys: the keys equal to T still
//        needed are taken lowest index first, each CTA taking what remains
//        after the ties of the CTAs before it (CTAs are in index order);
//   4. every CTA writes its chosen indices in ascending order at its offset
//      (the chosen counts of the CTAs before it) from a ballot bitmap.
// ---------------------------------------------------------------------------
constexpr int kTkThreads = 1024;
constexpr int kTkMaxCluster = 8;
constexpr int kTkDigit = 12;
constexpr int kTkBins = 1 << kTkDigit;
constexpr int kTkBlocks = 64;   // coarse blocks of a level's bins
constexpr int kTkCand = 256;    // candidates ranked directly

template <int PER>
struct TkLayout {
  static constexpr int kSlice = kTkThreads * PER;
  static constexpr int kWords = kSlice / 32;                 // at most one per thread
  static constexpr uint32_t KEYS = 0;                        // [kSlice]
  static constexpr uint32_t HIST = KEYS + kSlice * 4;        // [3 levels][4096]
  static constexpr uint32_t BLK = HIST + 3 * kTkBins * 4;    // [3 levels][64] block sums of this CTA
  static constexpr uint32_t FINE = BLK + 3 * kTkBlocks * 4;  // [64] cluster-summed bins of the picked block
  static constexpr uint32_t COARSE = FINE + 64 * 4;          // [64] cluster-summed block sums
  static constexpr uint32_t BM = COARSE + kTkBlocks * 4;     // chosen bitmap
  static constexpr uint32_t TB = BM + kWords * 4;            // tie bitmap
  static constexpr uint32_t TP = TB + kWords * 4;            // ties before each word
  static constexpr uint32_t XB = TP + kWords * 4;            // candidates chosen by rank
  static constexpr uint32_t CKEY = XB + kWords * 4;          // [256] this CTA's candidates: key
  static constexpr uint32_t CIDX = CKEY + kTkCand * 4;       // [256] and row index
  static constexpr uint32_t AKEY = CIDX + kTkCand * 4;       // [256] the cluster's candidates: key
  static constexpr uint32_t AIDX = AKEY + kTkCand * 4;       // [256] and row index
  static constexpr uint32_t MISC = AIDX + kTkCand * 4;
  static constexpr uint32_t SMEM = MISC + 1024;
  static_assert(kWords <= kTkThreads, "one bitmap word per thread");
};

// misc words
constexpr int kMiscRes = 32;      // [32..34] picked digit, count above it, count in it
constexpr int kMiscGt = 38;       // keys > T here
constexpr int kMiscTie = 39;      // keys == T here
constexpr int kMiscChosen = 40;   // chosen keys here
constexpr int kMiscCand = 41;     // candidates here
constexpr int kMiscBlk = 42;      // [42..43] picked block, count above it

// inclusive block-wide scan of one value per thread (1024 threads); warp_s[31] = total
__device__ __forceinline__ uint32_t block_scan_incl(uint32_t v, uint32_t* warp_s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  __syncthreads();
  if (lane == 31) warp_s[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_s[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += x;
    }
    warp_s[lane] = w;
  }
  __syncthreads();
  return v + (warp > 0 ? warp_s[warp - 1] : 0u);
}

// `local` in CTA r of the cluster; a plain shared-memory address when the
// cluster is one CTA (distributed shared memory is slower even for oneself)
template <typename T>
__device__ __forceinline__ T* tk_at(cg::cluster_group& cluster, T* local, uint32_t r, uint32_t C) {
  return C == 1 ? local : cluster.map_shared_rank(local, r);
}

// u32 at `local` in every CTA r < C of the cluster; all loads issued at once
__device__ __forceinline__ void cluster_gather_u32(cg::cluster_group& cluster, const uint32_t* local, uint32_t C,
                                                   uint32_t (&v)[kTkMaxCluster]) {
#pragma unroll
  for (int r = 0; r < kTkMaxCluster; ++r) v[r] = (uint32_t)r < C ? *tk_at(cluster, local, (uint32_t)r, C) : 0u;
}

__device__ __forceinline__ uint32_t cluster_sum_u32(cg::cluster_group& cluster, const uint32_t* local, uint32_t C) {
  uint32_t v[kTkMaxCluster];
  cluster_gather_u32(cluster, local, C, v);
  uint32_t s = 0;
#pragma unroll
  for (int r = 0; r < kTkMaxCluster; ++r) s += v[r];
  return s;
}

__device__ __forceinline__ void tk_sync(cg::cluster_group& cluster, uint32_t C) {
  if (C > 1) cluster.sync();
  else __syncthreads();
}

// The digit holding the need-th largest key of a level whose local histogram
// h has nb = 2^w bins (bin = digit). Stage 1 sums this CTA's 64 block sums
// (blk) over the cluster and picks a block; stage 2 sums that block's bins
// over the cluster and picks the bin. Leaves (digit, count above, count in
// it) in misc[kMiscRes..]; called by every thread of every CTA of the
// cluster, ends with the block synchronised.
__device__ __noinline__ void tk_pick(cg::cluster_group& cluster, uint32_t C, const uint32_t* h, uint32_t* blk,
                                     uint32_t* coarse, uint32_t* fine, int w, uint32_t need, uint32_t* misc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = 1 << w;
  const int n_blk = nb < kTkBlocks ? nb : kTkBlocks;
  const int bpb = nb / n_blk;  // bins per block, a power of two up to 64
  __syncthreads();  // this CTA's histogram is complete
  if (bpb >= 4) {
    const int g = bpb / 4;  // threads per block: 1 .. 16
    uint32_t v = 0;
    if (4 * tid < nb) {
      const uint4 x = *reinterpret_cast<const uint4*>(h + 4 * tid);
      v = x.x + x.y + x.z + x.w;
    }
    for (int o = 1; o < g; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (4 * tid < nb && (tid & (g - 1)) == 0) blk[tid / g] = v;
  } else if (tid < n_blk) {
    uint32_t v = 0;
    for (int j = 0; j < bpb; ++j) v += h[tid * bpb + j];
    blk[tid] = v;
  }
  tk_sync(cluster, C);  // every CTA's histogram and block sums are complete
  if (tid < n_blk) coarse[tid] = cluster_sum_u32(cluster, blk + tid, C);
  __syncthreads();
  // stage 1 (warp 0): lane l takes blocks n_blk-1-2l and n_blk-2-2l
  if (warp == 0) {
    const int b0 = n_blk - 1 - 2 * lane, b1 = b0 - 1;
    const uint32_t c0 = b0 >= 0 ? coarse[b0] : 0u, c1 = b1 >= 0 ? coarse[b1] : 0u;
    const uint32_t sum = c0 + c1;
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const uint32_t excl = incl - sum;
    if (excl < need && need <= incl) {
      const bool first = excl + c0 >= need;
      misc[kMiscBlk] = (uint32_t)(first ? b0 : b1);
      misc[kMiscBlk + 1] = first ? excl : excl + c0;
    }
  }
  __syncthreads();
  const int bsel = (int)misc[kMiscBlk];
  const uint32_t above_blk = misc[kMiscBlk + 1];
  // stage 2: the picked block's bins, top first
  if (tid < bpb) fine[tid] = cluster_sum_u32(cluster, h + bsel * bpb + (bpb - 1 - tid), C);
  __syncthreads();
  if (warp == 0) {
    const int i0 = 2 * lane, i1 = i0 + 1;  // positions from the top of the block
    const uint32_t c0 = i0 < bpb ? fine[i0] : 0u, c1 = i1 < bpb ? fine[i1] : 0u;
    const uint32_t sum = c0 + c1;
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const uint32_t excl = incl - sum;
    const uint32_t need2 = need - above_blk;
    if (excl < need2 && need2 <= incl) {
      const bool first = excl + c0 >= need2;
      const int pos = first ? i0 : i1;
      misc[kMiscRes] = (uint32_t)(bsel * bpb + (bpb - 1 - pos));
      misc[kMiscRes + 1] = above_blk + (first ? excl : excl + c0);
      misc[kMiscRes + 2] = first ? c0 : c1;
    }
  }
  __syncthreads();
}

// One-CTA form of the pick (no cluster): thread t owns bins nb-1-4t ..
// nb-4-4t of the local histogram and a block scan runs from the top digit
// down. Same result in misc[kMiscRes..]; ends with the block synchronised.
__device__ __noinline__ void tk_pick_local(const uint32_t* h, int w, uint32_t need, uint32_t* warp_s,
                                           uint32_t* misc) {
  const int tid = threadIdx.x;
  const int nb = 1 << w;
  __syncthreads();  // the histogram is complete
  uint32_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
  const int top = nb - 1 - 4 * tid;  // highest bin of this thread
  if (top >= 3) {
    const uint4 v = *reinterpret_cast<const uint4*>(h + top - 3);
    c0 = v.w;
    c1 = v.z;
    c2 = v.y;
    c3 = v.x;
  } else if (top >= 0) {
    c0 = h[top];
    if (top >= 1) c1 = h[top - 1];
    if (top >= 2) c2 = h[top - 2];
  }
  const uint32_t sum = c0 + c1 + c2 + c3;
  const uint32_t incl = block_scan_incl(sum, warp_s);
  const uint32_t excl = incl - sum;
  if (excl < need && need <= incl) {
    const uint32_t c[4] = {c0, c1, c2, c3};
    uint32_t run = excl;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (run + c[j] >= need) {
        misc[kMiscRes] = (uint32_t)(top - j);
        misc[kMiscRes + 1] = run;
        misc[kMiscRes + 2] = c[j];
        break;
      }
      run += c[j];
    }
  }
  __syncthreads();
}

enum TkMode { kTkAll = 0, kTkExact = 1, kTkCandRank = 2, kTkTies = 3 };

template <int PER>
__global__ void __launch_bounds__(kTkThreads, 1) topk_cluster_kernel(const float* __restrict__ scores, int64_t ld,
                                                                    const int32_t* __restrict__ n_vis,
                                                                    int64_t max_vis, int k,
                                                                    int32_t* __restrict__ out_idx) {
  using L = TkLayout<PER>;
  extern __shared__ __align__(16) unsigned char tk_smem[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(tk_smem + L::KEYS);
  uint32_t* hist = reinterpret_cast<uint32_t*>(tk_smem + L::HIST);
  uint32_t* blk = reinterpret_cast<uint32_t*>(tk_smem + L::BLK);
  uint32_t* fine = reinterpret_cast<uint32_t*>(tk_smem + L::FINE);
  uint32_t* coarse = reinterpret_cast<uint32_t*>(tk_smem + L::COARSE);
  uint32_t* bm = reinterpret_cast<uint32_t*>(tk_smem + L::BM);
  uint32_t* tb = reinterpret_cast<uint32_t*>(tk_smem + L::TB);
  uint32_t* tp = reinterpret_cast<uint32_t*>(tk_smem + L::TP);
  uint32_t* xb = reinterpret_cast<uint32_t*>(tk_smem + L::XB);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(tk_smem + L::CKEY);
  uint32_t* cidx = reinterpret_cast<uint32_t*>(tk_smem + L::CIDX);
  uint32_t* akey = reinterpret_cast<uint32_t*>(tk_smem + L::AKEY);
  uint32_t* aidx = reinterpret_cast<uint32_t*>(tk_smem + L::AIDX);
  uint32_t* misc = reinterpret_cast<uint32_t*>(tk_smem + L::MISC);
  uint32_t* warp_s = misc;

  pdl_wait();  // the scores of the previous kernel
  pdl_trigger();
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t rank = cluster.block_rank();
  const uint32_t C = cluster.num_blocks();
  const int q = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = (int)min((int64_t)max(n_vis[q], 0), max_vis);
  const int64_t base = (int64_t)rank * L::kSlice;
  const int cnt = (int)max((int64_t)0, min((int64_t)L::kSlice, (int64_t)nv - base));
  const uint32_t need = (uint32_t)min(k, nv);
  const bool all = (uint32_t)nv <= need;  // every visible entry is chosen (uniform over the cluster)

  // ---- slice -> keys; histograms, rank bitmap and counters zeroed meanwhile
  {
    const float* row = scores + (int64_t)q * ld + base;
    float v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int li = u * kTkThreads + tid;
      v[u] = li < cnt ? row[li] : 0.f;
    }
    uint4* h4 = reinterpret_cast<uint4*>(hist);
    for (int i = tid; i < 3 * kTkBins / 4; i += kTkThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < L::kWords) xb[tid] = 0u;
    if (tid == 0) {
      misc[kMiscGt] = 0u;
      misc[kMiscTie] = 0u;
      misc[kMiscCand] = 0u;
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) keys[u * kTkThreads + tid] = score_key(v[u]);
  }
  __syncthreads();

  // state after the search: keys whose top (32 - shift) bits are > P are
  // chosen; of those equal to P: all (exact), the ones marked in xb (rank),
  // or, with shift == 0, the first take_t in index order (ties)
  uint32_t P = 0, take_t = 0;
  int shift = 32;
  int mode = all ? kTkAll : kTkTies;
  if (!all) {
    // the digits start at the top bit (finding the cluster's common prefix
    // first, one more cluster-wide exchange, measured slower)
    shift = 32;
    P = 0u;
    uint32_t rem = need;
    // ---- digit levels
#pragma unroll 1
    for (int lvl = 0; shift > 0; ++lvl) {
      const int w = min(kTkDigit, shift);
      const int sh = shift - w;
      const uint32_t dmask = (1u << w) - 1u;
      uint32_t* h = hist + kTkBins * lvl;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const uint32_t x = keys[u * kTkThreads + tid];
        const bool ok = u * kTkThreads + tid < cnt && (shift >= 32 || (x >> shift) == P);
        if (ok) atomicAdd(&h[(x >> sh) & dmask], 1u);
      }
      if (C == 1) tk_pick_local(h, w, rem, warp_s, misc);
      else tk_pick(cluster, C, h, blk + kTkBlocks * lvl, coarse, fine, w, rem, misc);
      P = (shift >= 32 ? 0u : (P << w)) | misc[kMiscRes];
      rem -= misc[kMiscRes + 1];
      const uint32_t at = misc[kMiscRes + 2];
      shift = sh;
      __syncthreads();  // misc[kMiscRes..] is rewritten by the next level
      if (at == rem) {
        mode = kTkExact;
        break;
      }
      // across a cluster a few candidates are ranked at once; one CTA goes
      // on with another level, which is cheaper there
      if (C > 1 && at <= (uint32_t)kTkCand) {
        mode = kTkCandRank;
        break;
      }
    }
    take_t = rem;
  }
  // ---- rank path: the keys whose top bits equal P (at most 256 over the
  // cluster) are gathered and each CTA ranks its own against all of them
  if (mode == kTkCandRank) {
    // candidate bitmap (word w = u*32 + warp), then slots in index order from
    // a block scan of the words' counts; no shared counter
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int li = u * kTkThreads + tid;
      const uint32_t x = keys[li];
      const uint32_t bal = __ballot_sync(0xffffffffu, li < cnt && (x >> shift) == P);
      if (lane == 0) tb[u * 32 + warp] = bal;
    }
    __syncthreads();
    {
      const uint32_t cw = tid < L::kWords ? tb[tid] : 0u;  // thread tid owns word tid
      uint32_t slot = block_scan_incl(__popc(cw), warp_s) - __popc(cw);
      if (tid == 0) misc[kMiscCand] = warp_s[31];
      uint32_t bits = cw;
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1u;
        if (slot < (uint32_t)kTkCand) {
          const uint32_t li = 32u * (uint32_t)tid + (uint32_t)bit;
          ckey[slot] = keys[li];
          cidx[slot] = (uint32_t)base + li;
        }
        ++slot;
      }
    }
    tk_sync(cluster, C);  // every CTA's candidate list is complete
    uint32_t cn[kTkMaxCluster];
    cluster_gather_u32(cluster, misc + kMiscCand, C, cn);
    uint32_t n_all = 0, start = 0, src = 0;
#pragma unroll
    for (int r = 0; r < kTkMaxCluster; ++r) {
      const uint32_t c = min(cn[r], (uint32_t)kTkCand);
      if ((uint32_t)tid >= n_all && (uint32_t)tid < n_all + c) {
        src = (uint32_t)r;
        start = n_all;
      }
      n_all += c;
    }
    n_all = min(n_all, (uint32_t)kTkCand);
    if ((uint32_t)tid < n_all) {
      const uint32_t j = (uint32_t)tid - start;
      akey[tid] = *tk_at(cluster, ckey + j, src, C);
      aidx[tid] = *tk_at(cluster, cidx + j, src, C);
    }
    __syncthreads();
    const uint32_t n_mine = min(misc[kMiscCand], (uint32_t)kTkCand);
    {
      // four threads per candidate (1024 / 256), each over every fourth
      // entry; the four partial ranks meet by shuffles within the warp
      const uint32_t i = (uint32_t)tid >> 2, part = (uint32_t)tid & 3u;
      const bool mine = i < n_mine;
      const uint32_t kx = mine ? ckey[i] : 0u, ix = mine ? cidx[i] : 0u;
      uint32_t rk = 0;
      if (mine) {
#pragma unroll 4
        for (uint32_t j = part; j < n_all; j += 4) {
          const uint32_t ky = akey[j], iy = aidx[j];
          rk += (ky > kx || (ky == kx && iy < ix)) ? 1u : 0u;
        }
      }
      rk += __shfl_xor_sync(0xffffffffu, rk, 1);
      rk += __shfl_xor_sync(0xffffffffu, rk, 2);
      if (mine && part == 0 && rk < take_t) {
        const uint32_t li = ix - (uint32_t)base;
        atomicOr(&xb[li >> 5], 1u << (li & 31u));
      }
    }
    __syncthreads();
  }
  // ---- ties at T = P (shift == 0, more ties than 256): counts above T and
  // at T here, exchanged once across the cluster; this CTA may take the ties
  // that the CTAs before it leave, lowest index first
  uint32_t quota = 0, off = 0;
  bool off_known = false;
  if (mode == kTkAll) {
    off = (uint32_t)base;  // every earlier CTA is full and fully chosen
    off_known = true;
  } else if (mode == kTkTies) {
    uint32_t ngt = 0, nt = 0;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int li = u * kTkThreads + tid;
      const uint32_t x = keys[li];
      const uint32_t bt = __ballot_sync(0xffffffffu, li < cnt && x == P);
      const uint32_t bg = __ballot_sync(0xffffffffu, li < cnt && x > P);
      if (lane == 0) tb[u * 32 + warp] = bt;
      nt += __popc(bt);
      ngt += __popc(bg);
    }
    if (lane == 0) {
      atomicAdd(&misc[kMiscGt], ngt);
      atomicAdd(&misc[kMiscTie], nt);
    }
    tk_sync(cluster, C);
    uint32_t g[kTkMaxCluster], t[kTkMaxCluster];
    cluster_gather_u32(cluster, misc + kMiscGt, C, g);
    cluster_gather_u32(cluster, misc + kMiscTie, C, t);
    uint32_t ties_before = 0;
#pragma unroll
    for (int r = 0; r < kTkMaxCluster; ++r) {
      if ((uint32_t)r < rank) {
        const uint32_t qr = take_t > ties_before ? min(t[r], take_t - ties_before) : 0u;
        off += g[r] + qr;
        ties_before += t[r];
      }
    }
    off_known = true;
    quota = take_t > ties_before ? take_t - ties_before : 0u;
    if (quota > 0) {
      const uint32_t tw = tid < L::kWords ? tb[tid] : 0u;  // thread tid owns word tid
      const uint32_t pre = block_scan_incl(__popc(tw), warp_s) - __popc(tw);
      if (tid < L::kWords) tp[tid] = pre;
      __syncthreads();
    }
  }
  // ---- chosen bitmap
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int li = u * kTkThreads + tid;
    const int w = u * 32 + warp;
    const uint32_t x = keys[li];
    bool chosen;
    if (mode == kTkAll) {
      chosen = li < cnt;
    } else if (mode == kTkExact) {
      chosen = li < cnt && (x >> shift) >= P;
    } else if (mode == kTkCandRank) {
      chosen = li < cnt && ((x >> shift) > P || ((xb[w] >> lane) & 1u) != 0u);
    } else {
      chosen = li < cnt && x > P;
      if (li < cnt && x == P && quota > 0)
        chosen = tp[w] + __popc(tb[w] & ((1u << lane) - 1u)) < quota;
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, chosen);
    if (lane == 0) bm[w] = bal;
  }
  __syncthreads();
  // ---- offsets of the words (thread tid owns word tid) and of this CTA
  const uint32_t wbits = tid < L::kWords ? bm[tid] : 0u;
  const uint32_t pre = block_scan_incl(__popc(wbits), warp_s) - __popc(wbits);
  if (!off_known && C > 1) {
    if (tid == 0) misc[kMiscChosen] = warp_s[31];
    cluster.sync();
    uint32_t c[kTkMaxCluster];
    cluster_gather_u32(cluster, misc + kMiscChosen, C, c);
#pragma unroll
    for (int r = 0; r < kTkMaxCluster; ++r)
      if ((uint32_t)r < rank) off += c[r];
  }
  // ---- chosen indices, ascending, at this CTA's offset
  {
    int32_t* o = out_idx + (int64_t)q * k;
    if (tid < L::kWords) {
      const int64_t li0 = base + 32 * (int64_t)tid;
      uint32_t bits = wbits, pos = off + pre;
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1u;
        if (pos < (uint32_t)k) o[pos] = (int32_t)(li0 + bit);
        ++pos;
      }
    }
    if (rank == 0)
      for (int i = (int)need + tid; i < k; i += kTkThreads) o[i] = -1;
  }
  // keep every CTA's shared memory alive until all remote reads are done
  if (C > 1) cluster.sync();
}

static int topk_cluster_size(int64_t max_vis, int slice) {
  const int64_t c = (max_vis + slice - 1) / slice;
  return (int)(c < 1 ? 1 : c);
}

// The candidate region of the workspace (after the histograms and counts):
// the three-launch path's (key, index) candidates, or the sliced path's
// per-slice lists (n_query x slices x k entry indices, fewer bytes).
static size_t topk_lists_offset(int n_query) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)n_query * kHistBins * 4) + al((size_t)n_query * 4);
}

size_t topk_workspace_bytes(int n_query, int64_t max_vis) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)n_query * kHistBins * 4) + al((size_t)n_query * 4) +
         al((size_t)n_query * (size_t)(max_vis > 0 ? max_vis : 1) * 8);
}

// ---------------------------------------------------------------------------
// Rows of at most TPB * PER scores: one CTA per query, no cluster. Thread t
// keeps the order-preserving keys of entries PER t .. PER t + PER - 1 in
// registers. The search narrows the threshold eleven bits at a time from
// the top: one CTA-wide histogram of the keys still in play (plain shared
// atomics), a block scan over its bins finds the one that holds the k-th
// largest, and the search stops once that bin holds exactly the keys still
// needed, or when no bits are left (ties at one key value, taken in index
// order). With 24 keys a thread (rows of up to 6,144) the kernel is held to
// 64 registers, so that four CTAs share an SM instead of three (chunked
// prefill step 960 -> 950 us); with 8 keys the bound measured slower. (Finding the row's common prefix first, or 8-bit digits in per-warp
// histograms, measured slower.) One 64-bit block scan of
// (above-threshold, at-threshold) counts then gives every thread the output
// positions of its entries, which come out in ascending index order.
// map set: entry e of the row is pool position e, written out as the entry
// index (map[q, e >> map_shift] << map_shift) | (e & (2^map_shift - 1))
struct TkMap {
  const int32_t* blocks = nullptr;
  int ld = 0;
  int shift = 0;
  int base = 0;  // without blocks: entry = base + e (a slice of a longer row)
  __device__ __forceinline__ int32_t operator()(int q, int e) const {
    if (blocks == nullptr) return base + e;
    return (blocks[(int64_t)q * ld + (e >> shift)] << shift) | (e & ((1 << shift) - 1));
  }
};

// This thread's keys: entries PER t .. PER t + PER - 1 of the row as
// order-preserving keys (0, below every score's key, past n).
template <int PER>
__device__ __forceinline__ void row_load_keys(const float* __restrict__ row, const float* __restrict__ scores, int64_t ld,
                                              int e0, int n, uint32_t (&key)[PER]) {
  if (((ld & 3) == 0) && ((reinterpret_cast<uintptr_t>(scores) & 15) == 0) && e0 + PER <= n) {
#pragma unroll
    for (int c = 0; c < PER / 4; ++c) {
      const float4 v = reinterpret_cast<const float4*>(row + e0)[c];
      key[4 * c] = score_key(v.x);
      key[4 * c + 1] = score_key(v.y);
      key[4 * c + 2] = score_key(v.z);
      key[4 * c + 3] = score_key(v.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < PER; ++i) key[i] = (e0 + i < n) ? score_key(row[e0 + i]) : 0u;
  }
}

// Threshold search over the keys in play, eleven bits a level from the top
// key bit: one CTA-wide histogram of the keys still in play (plain shared
// atomics), a block scan over its bins finds the one that holds the k-th
// largest key, and the search stops once that bin holds exactly the keys
// still needed, or when no bits are left (ties at one key value). On return
// the chosen entries are those with (key >> hi) > P, then `need` of those with
// (key >> hi) == P in index order (all of them when exact).
template <int TPB, int PER>
__device__ __forceinline__ void row_radix_search(const uint32_t (&key)[PER], int e0, int n, uint32_t k,
                                                 uint32_t* hist, uint32_t* res, uint32_t* wtot, uint32_t& P, int& hi,
                                                 uint32_t& need, bool& exact) {
  constexpr int NW = TPB / 32;
  constexpr int DB = 11;        // digit bits a level
  constexpr int NB = 1 << DB;
  constexpr int BPT = NB / TPB;  // bins a thread owns in the scan
  static_assert(NB % TPB == 0 && TPB % 32 == 0, "bins split evenly");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  hi = 32;
  P = 0u;
  need = k;
  exact = false;
  while (hi > 0) {
    const int lo = hi > DB ? hi - DB : 0;
    const int w = hi - lo;
    const uint32_t dmask = (1u << w) - 1u;
    const int nb = 1 << w;
    // the previous level read hist before its scan barriers and res after
    // its last one; both are rewritten only after the barriers below
    for (int i = tid; i < nb; i += TPB) hist[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (e0 + i < n && (hi >= 32 || (key[i] >> hi) == P)) atomicAdd(&hist[(key[i] >> lo) & dmask], 1u);
    __syncthreads();
    // thread t owns bins nb-1-BPT t .. nb-BPT (t+1), in descending order
    uint32_t c[BPT], sl = 0;
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
      const int bin = nb - 1 - (BPT * tid + b);
      c[b] = bin >= 0 ? hist[bin] : 0u;
      sl += c[b];
    }
    uint32_t incl = sl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const uint32_t own = lane < NW ? wtot[lane] : 0u;
      uint32_t t = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += v;
      }
      if (lane < NW) wtot[lane] = t - own;
    }
    __syncthreads();
    incl += wtot[warp];
    const uint32_t excl = incl - sl;
    if (excl < need && need <= incl) {
      // the first of this thread's bins where the running count reaches need
      // (predicated selects keep c[] in registers)
      uint32_t cum = excl, pick = BPT - 1, at = c[BPT - 1], before = excl;
      bool found = false;
#pragma unroll
      for (int b = 0; b < BPT; ++b) {
        const bool here = !found && cum + c[b] >= need;
        pick = here ? (uint32_t)b : pick;
        at = here ? c[b] : at;
        before = here ? cum : before;
        found = found || here;
        cum += c[b];
      }
      res[0] = (uint32_t)(nb - 1 - BPT * tid) - pick;
      res[1] = at;
      res[2] = before;
    }
    __syncthreads();
    const uint32_t bstar = res[0], nbin = res[1], above = res[2];
    need -= above;
    P = (hi >= 32 ? 0u : (P << w)) | bstar;
    hi = lo;
    if (nbin == need) {
      exact = true;
      break;
    }
  }
}

// Writes the chosen entries of the row in ascending index order: every
// entry with gt(key), then, in index order, `need` of those with eq(key)
// (all of them when exact). One 64-bit block scan of (above, at) counts
// gives each thread the output positions of its consecutive entries.
template <int TPB, int PER, class Gt, class Eq>
__device__ __forceinline__ void row_emit(const uint32_t (&key)[PER], int e0, int n, uint32_t need, bool exact, Gt gt,
                                         Eq eq, unsigned long long* wsum, int32_t* out, const TkMap& map, int q) {
  constexpr int NW = TPB / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (exact) {
    // every tie is taken (the common case): one 32-bit count of the chosen
    // keys and its block scan place them
    uint32_t n_ch = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) n_ch += (e0 + i < n && (gt(key[i]) || eq(key[i]))) ? 1u : 0u;
    uint32_t v = n_ch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
      uint32_t w = lane < NW ? (uint32_t)wsum[lane] : 0u;
      const uint32_t own = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += u;
      }
      if (lane < NW) wsum[lane] = w - own;  // exclusive over warps
    }
    __syncthreads();
    uint32_t pos = (uint32_t)wsum[warp] + v - n_ch;  // exclusive over threads
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (e0 + i < n && (gt(key[i]) || eq(key[i]))) out[pos++] = map(q, e0 + i);
    return;
  }
  uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (e0 + i < n) {
      n_gt += gt(key[i]) ? 1u : 0u;
      n_eq += eq(key[i]) ? 1u : 0u;
    }
  unsigned long long v = ((unsigned long long)n_eq << 32) | n_gt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < NW ? wsum[lane] : 0ull;
    const unsigned long long own = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < NW) wsum[lane] = w - own;  // exclusive over warps
  }
  __syncthreads();
  v += wsum[warp] - (((unsigned long long)n_eq << 32) | n_gt);  // exclusive over threads
  const uint32_t gt_before = (uint32_t)(v & 0xFFFFFFFFull), eq_before = (uint32_t)(v >> 32);
  uint32_t pos, eq_left;
  if (exact) {
    pos = gt_before + eq_before;
    eq_left = n_eq;
  } else {
    pos = gt_before + min(eq_before, need);
    eq_left = need > eq_before ? min(n_eq, need - eq_before) : 0u;
  }
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (e0 + i < n) {
      bool take = gt(key[i]);
      if (eq(key[i]) && eq_left > 0) {
        take = true;
        --eq_left;
      }
      if (take) out[pos++] = map(q, e0 + i);
    }
}

template <int TPB, int PER>
__global__ void __launch_bounds__(TPB, (PER == 24 ? 4 : 1)) topk_row_kernel(const float* __restrict__ scores, int64_t ld,
                                                      const int32_t* __restrict__ n_vis, int64_t max_vis, int k,
                                                      int32_t* __restrict__ out_idx, const TkMap map) {
  constexpr int NW = TPB / 32;
  static_assert(PER % 4 == 0, "float4 loads");
  __shared__ uint32_t hist[1 << 11];
  __shared__ uint32_t res[3];
  __shared__ uint32_t wtot[NW];
  __shared__ unsigned long long wsum[NW];
  pdl_wait();  // the scores (and pool counts) of the previous kernel
  pdl_trigger();
  const int tid = threadIdx.x;
  const int q = blockIdx.x;
  const int n = (int)min((int64_t)max(n_vis[q], 0), max_vis);
  int32_t* out = out_idx + (int64_t)q * k;
  if (n <= k) {
    for (int i = tid; i < k; i += TPB) out[i] = i < n ? map(q, i) : -1;
    return;
  }
  const float* row = scores + (int64_t)q * ld;
  const int e0 = PER * tid;
  uint32_t key[PER];
  row_load_keys<PER>(row, scores, ld, e0, n, key);
  uint32_t P, need;
  int hi;
  bool exact;
  row_radix_search<TPB, PER>(key, e0, n, (uint32_t)k, hist, res, wtot, P, hi, need, exact);
  row_emit<TPB, PER>(key, e0, n, need, exact, [&](uint32_t x) { return (x >> hi) > P; },
                     [&](uint32_t x) { return (x >> hi) == P; }, wsum, out, map, q);
}

// The decode form for rows of up to 16,384 scores held by 1,024 threads
// (few queries, one CTA each; the whole step waits on the slowest row).
// Scores near the top sit close to the row's largest key M in key space, so
// the first level bins the distance d = M - key of every key within 2^24 of
// M (4,096 bins of 2^12, bin 0 the top; for positive scores that is about
// two binades below the largest): only keys near the top touch the
// histogram, which keeps shared-atomic contention low, and one warp scans
// the bins, so the level costs two barriers. A second level bins the low 12
// bits of d inside the picked bin, which pins the threshold key exactly;
// ties at it are taken in index order. Rows whose k largest keys do not all
// lie within 2^24 of M fall back to the radix search above.
constexpr int kRelBins = 4096;
constexpr int kRelShift = 12;
constexpr int kRelSub = 1 << kRelShift;

// The bin of h (NB bins, bin 0 the top) where the count from the top reaches
// need, in two stages without a serial walk: every warp sums one group of
// NB / 32 bins (four per lane, then a warp sum); after a barrier, warp 0
// scans the 32 group sums, picks the group, scans that group's bins four per
// lane and picks the bin. Leaves res = (bin, count above it, count in it),
// or res[0] = ~0 if the bins hold fewer than need. Called by all 1,024
// threads; ends without a barrier (the caller synchronises before reading).
template <int NB>
__device__ __forceinline__ void rel_pick(const uint32_t* h, uint32_t need, uint32_t* res, uint32_t* gsum) {
  constexpr int G = NB / 32;  // bins a group (one per warp)
  static_assert(G == 128, "four bins a lane");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    const uint4 v = reinterpret_cast<const uint4*>(h + G * warp)[lane];
    uint32_t x = v.x + v.y + v.z + v.w;
    x = __reduce_add_sync(0xffffffffu, x);
    if (lane == 0) gsum[warp] = x;
  }
  __syncthreads();
  if (warp != 0) return;
  const uint32_t s = gsum[lane];
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const uint32_t reach = __ballot_sync(0xffffffffu, incl >= need);
  if (reach == 0u) {
    if (lane == 0) res[0] = 0xFFFFFFFFu;
    return;
  }
  const int g = __ffs(reach) - 1;
  const uint32_t above_g = __shfl_sync(0xffffffffu, incl - s, g);
  const uint4 v = reinterpret_cast<const uint4*>(h + G * g)[lane];
  const uint32_t c4 = v.x + v.y + v.z + v.w;
  uint32_t inc2 = c4;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, inc2, o);
    if (lane >= o) inc2 += u;
  }
  const uint32_t need2 = need - above_g;
  const uint32_t reach2 = __ballot_sync(0xffffffffu, inc2 >= need2);
  if (lane == __ffs(reach2) - 1) {
    uint32_t cum = above_g + inc2 - c4;
    const uint32_t c[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (cum + c[j] >= need) {
        res[0] = (uint32_t)(G * g + 4 * lane + j);
        res[1] = cum;
        res[2] = c[j];
        break;
      }
      cum += c[j];
    }
  }
}

// n_slices > 1: CTA (q, s) = (blockIdx.x / n_slices, blockIdx.x % n_slices)
// selects among entries [s * 16,384, (s + 1) * 16,384) of row q only and
// writes that slice's k largest (entry indices of the whole row) to list
// out_idx[(q * n_slices + s) * k ..]; topk_merge_kernel then merges the lists.
template <int PER>
__global__ void __launch_bounds__(1024) topk_row_rel_kernel(const float* __restrict__ scores, int64_t ld,
                                                           const int32_t* __restrict__ n_vis, int64_t max_vis, int k,
                                                           int32_t* __restrict__ out_idx, TkMap map,
                                                           int n_slices = 1) {
  constexpr int TPB = 1024, NW = 32;
  static_assert(PER % 4 == 0, "float4 loads");
  __shared__ __align__(16) uint32_t h1[kRelBins];
  __shared__ __align__(16) uint32_t h2[kRelSub];  // also the fallback's histogram
  __shared__ uint32_t res[3];
  __shared__ uint32_t wtot[NW];
  __shared__ unsigned long long wsum[NW];
  __shared__ uint32_t s_max;
  __shared__ uint32_t gsum[32];
  pdl_wait();  // the scores of the previous kernel
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31;
  const int q = blockIdx.x / n_slices, sl = blockIdx.x % n_slices;
  constexpr int kSlice = TPB * PER;
  const int64_t s0 = (int64_t)sl * kSlice;
  const int n = (int)max((int64_t)0, min(min((int64_t)max(n_vis[q], 0), max_vis) - s0, (int64_t)kSlice));
  map.base = (int)s0;
  int32_t* out = out_idx + (int64_t)blockIdx.x * k;
  if (n <= k) {
    for (int i = tid; i < k; i += TPB) out[i] = i < n ? map(q, i) : -1;
    return;
  }
  const float* row = scores + (int64_t)q * ld + s0;
  const int e0 = PER * tid;
  uint32_t key[PER];
  row_load_keys<PER>(row, scores, ld, e0, n, key);
  // histograms zeroed and the row's largest key found meanwhile
  {
    uint4* z1 = reinterpret_cast<uint4*>(h1);
    uint4* z2 = reinterpret_cast<uint4*>(h2);
    for (int i = tid; i < kRelBins / 4; i += TPB) z1[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < kRelSub / 4; i += TPB) z2[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid == 0) s_max = 0u;
  uint32_t mx = 0u;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (e0 + i < n) mx = max(mx, key[i]);
  mx = __reduce_max_sync(0xffffffffu, mx);
  __syncthreads();
  if (lane == 0) atomicMax(&s_max, mx);
  __syncthreads();
  const uint32_t M = s_max;
  // level 1: distance to the top in bins of 2^12 key steps
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const uint32_t d = M - key[i];
    if (e0 + i < n && d < ((uint32_t)kRelBins << kRelShift)) atomicAdd(&h1[d >> kRelShift], 1u);
  }
  __syncthreads();
  rel_pick<kRelBins>(h1, (uint32_t)k, res, gsum);
  __syncthreads();
  const uint32_t b1 = res[0];
  // every path ends with one threshold D on d = M - key: the entries with
  // d < D, then `need` of those with d == D in index order (all if exact)
  uint32_t D, need;
  bool exact;
  if (b1 == 0xFFFFFFFFu) {
    // the k largest keys reach further than 2^24 below the top: the radix
    // search from the top bit (chosen: key >= P << hi when exact, else
    // key > P and ties at P)
    __syncthreads();  // every thread has read res[0]
    uint32_t P;
    int hi;
    row_radix_search<TPB, PER>(key, e0, n, (uint32_t)k, h2, res, wtot, P, hi, need, exact);
    D = exact ? M - (P << hi) : M - P;
  } else if (res[2] == (uint32_t)k - res[1]) {
    // every key of the picked bin is needed: d up to the bin's last step
    D = ((b1 + 1u) << kRelShift) - 1u;
    need = 0u;
    exact = true;
  } else {
    // level 2: the low 12 bits of d inside the picked bin pin the threshold
    const uint32_t need1 = (uint32_t)k - res[1];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const uint32_t d = M - key[i];
      if (e0 + i < n && (d >> kRelShift) == b1) atomicAdd(&h2[d & (kRelSub - 1)], 1u);
    }
    __syncthreads();
    rel_pick<kRelSub>(h2, need1, res, gsum);
    __syncthreads();
    D = (b1 << kRelShift) | res[0];  // the threshold key is M - D
    need = need1 - res[1];
    exact = res[2] == need;
  }
  row_emit<TPB, PER>(key, e0, n, need, exact, [&](uint32_t x) { return M - x < D; },
                     [&](uint32_t x) { return M - x == D; }, wsum, out, map, q);
}

template <int TPB, int PER>
static cudaError_t launch_topk_row(cudaStream_t st, int n_query, const float* scores, int64_t ld,
                                   const int32_t* n_vis, int64_t max_vis, int k, int32_t* out_idx,
                                   const TkMap& map, bool pdl) {
  const cudaError_t e = launch_ex(topk_row_kernel<TPB, PER>, dim3(n_query), dim3(TPB), 0, st, pdl, 0, scores, ld,
                                  n_vis, max_vis, k, out_idx, map);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The hierarchical indexer's block scores: the largest score among each
// block's visible entries; the block holding entry n_vis - 1 (still filling)
// scores +inf so that the block top-k keeps it. nb[q] = the number of blocks.
__global__ void __launch_bounds__(256) block_max_kernel(const float* __restrict__ scores, int64_t ld,
                                                        const int32_t* __restrict__ n_vis, int64_t max_vis,
                                                        int shift, float* __restrict__ bscore, int64_t ld_b,
                                                        int32_t* __restrict__ nb_out) {
  const int q = blockIdx.y;
  const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const int64_t n = min((int64_t)max(n_vis[q], 0), max_vis);
  const int64_t nb = (n + (1 << shift) - 1) >> shift;
  if (blockIdx.x == 0 && threadIdx.x == 0) nb_out[q] = (int32_t)nb;
  if (b >= nb) return;
  const float* row = scores + (int64_t)q * ld + (b << shift);
  const int lim = (int)min((int64_t)1 << shift, n - (b << shift));
  float mx = row[0];
  for (int i = 1; i < lim; ++i) mx = fmaxf(mx, row[i]);
  bscore[(int64_t)q * ld_b + b] = (b == nb - 1) ? INFINITY : mx;
}

size_t candidate_pool_workspace_bytes(int n_query, int64_t max_vis, int shift) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const int64_t ld_b = max((int64_t)1, (max_vis + (1 << shift) - 1) >> shift);
  return al((size_t)n_query * ld_b * 4) + al((size_t)n_query * 4) + al(topk_workspace_bytes(n_query, ld_b));
}

cudaError_t launch_candidate_pool(cudaStream_t st, int n_query, const float* scores, int64_t ld,
                                  const int32_t* n_vis, int64_t max_vis, int shift, int keep, int32_t* cand,
                                  void* ws, int* n_launch) {
  if (n_query == 0) return cudaSuccess;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const int64_t ld_b = max((int64_t)1, (max_vis + (1 << shift) - 1) >> shift);
  char* p = reinterpret_cast<char*>(ws);
  float* bscore = reinterpret_cast<float*>(p);
  p += al((size_t)n_query * ld_b * 4);
  int32_t* nb = reinterpret_cast<int32_t*>(p);
  p += al((size_t)n_query * 4);
  const dim3 g((unsigned)((ld_b + 255) / 256), (unsigned)n_query);
  block_max_kernel<<<g, 256, 0, st>>>(scores, ld, n_vis, max_vis, shift, bscore, ld_b, nb);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *n_launch += 1;
  return launch_topk(st, n_query, bscore, ld_b, nb, ld_b, keep, cand, p, n_launch);
}

template <int PER>
static cudaError_t launch_topk_cluster(cudaStream_t st, int csize, int n_query, const float* scores, int64_t ld,
                                      const int32_t* n_vis, int64_t max_vis, int k, int32_t* out_idx, bool* launched,
                                      bool pdl) {
  *launched = false;
  const void* fn = (const void*)topk_cluster_kernel<PER>;
  const uint32_t smem = TkLayout<PER>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(n_query * csize));
  cfg.blockDim = dim3(kTkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg);
  cudaLaunchAttribute attr2[2] = {attr[0], attr[0]};
  if (pdl) {
    attr2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr2[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr2;
    cfg.numAttrs = 2;
  }
  if (e != cudaSuccess || max_clusters < 1) {
    cudaGetLastError();  // cluster shape not schedulable here: the caller takes the global-memory path
    return cudaSuccess;
  }
  // More queries than clusters resident at once: every query, however short,
  // would hold csize SMs for a whole selection, wave after wave. The
  // global-memory path spreads the work by each row's own length instead.
  if (n_query > max_clusters) return cudaSuccess;
  e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel<PER>, scores, ld, n_vis, max_vis, k, out_idx);
  if (e != cudaSuccess) return e;
  *launched = true;
  return cudaGetLastError();
}

cudaError_t launch_topk(cudaStream_t st, int n_query, const float* scores, int64_t ld, const int32_t* n_vis,
                        int64_t max_vis, int k, int32_t* out_idx, void* ws, int* n_launch, const int32_t* map_blocks,
                        int map_ld, int map_shift, bool pdl) {
  if (n_query == 0) return cudaSuccess;
  TkMap map;
  map.blocks = map_blocks;
  map.ld = map_ld;
  map.shift = map_shift;
  // rows of up to 16,384 scores: one CTA per query holding its row in registers
  if (max_vis <= 16384) {
    cudaError_t e;
    // the fewest keys a thread that fit: registers set how many rows an SM
    // holds at once (chunked prefill has thousands of rows of up to 6,144)
    if (max_vis <= 2048) e = launch_topk_row<256, 8>(st, n_query, scores, ld, n_vis, max_vis, k, out_idx, map, pdl);
    else if (max_vis <= 4096)
      e = launch_topk_row<256, 16>(st, n_query, scores, ld, n_vis, max_vis, k, out_idx, map, pdl);
    else if (max_vis <= 6144)
      e = launch_topk_row<256, 24>(st, n_query, scores, ld, n_vis, max_vis, k, out_idx, map, pdl);
    else if (max_vis <= 8192)
      e = launch_topk_row<256, 32>(st, n_query, scores, ld, n_vis, max_vis, k, out_idx, map, pdl);
    else {
      e = launch_ex(topk_row_rel_kernel<16>, dim3(n_query), dim3(1024), 0, st, pdl, 0, scores, ld, n_vis, max_vis, k,
                    out_idx, map, 1);
      if (e == cudaSuccess) e = cudaGetLastError();
    }
    if (e == cudaSuccess) *n_launch += 1;
    return e;
  }
  if (map_blocks != nullptr) return cudaErrorInvalidValue;  // pools hold at most 16,384 entries
  // a cluster of up to 8 CTAs per query, each holding 16,384 scores (a
  // 64K-context decode row is one CTA), or 32,768 for rows up to 262,144
  const int c16 = topk_cluster_size(max_vis, TkLayout<16>::kSlice);
  const int c32 = topk_cluster_size(max_vis, TkLayout<32>::kSlice);
  if (c32 <= kTkMaxCluster) {
    bool launched = false;
    cudaError_t e = c16 <= kTkMaxCluster
                        ? launch_topk_cluster<16>(st, c16, n_query, scores, ld, n_vis, max_vis, k, out_idx, &launched, pdl)
                        : launch_topk_cluster<32>(st, c32, n_query, scores, ld, n_vis, max_vis, k, out_idx, &launched,
                                                  pdl);
    if (e != cudaSuccess) return e;
    if (launched) {
      *n_launch += 1;
      return cudaSuccess;
    }
  }
  // More queries than clusters fit (ragged serving batches): each
  // 16,384-score slice selects its own k largest in one CTA (the decode form
  // above; slices past a row's end exit at once), and one CTA per query
  // merges the slices' lists with the tie rule, reading the scores by entry. A slice
  // list holds the k largest of the slice, so the row's k largest are among
  // the lists' union.
  {
    constexpr int kSliceLen = 1024 * 16;
    const int64_t n_slices = (max_vis + kSliceLen - 1) / kSliceLen;
    if (n_slices * k <= kSelCap) {
      int32_t* lists = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + topk_lists_offset(n_query));
      cudaError_t e = launch_ex(topk_row_rel_kernel<16>, dim3((unsigned)(n_query * n_slices)), dim3(1024), 0, st, pdl, 0,
                                scores, ld, n_vis, max_vis, k, lists, map, (int)n_slices);
      if (e == cudaSuccess) e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      const size_t smem = (size_t)kSelCap * 8 + (size_t)kMaxTopk * 4;
      e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        e = launch_ex(topk_merge_kernel, dim3((unsigned)n_query), dim3(1024), smem, st, pdl, 0, n_query, (int)n_slices,
                      k, (const float*)nullptr, (const int32_t*)lists, k, out_idx, scores, ld);
      if (e == cudaSuccess) e = cudaGetLastError();
      if (e == cudaSuccess) *n_launch += 2;
      return e;
    }
  }
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
