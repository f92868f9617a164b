// Lightning-indexer scores on the tensor cores, for many queries per sequence
// (chunked prefill): sigma_q(j) = sum_h w_{q,h} relu(q^I_{q,h} . k^I_j)
// ("Reading Notes of DeepSeek-V4.1-Flash", section 3f, C2 step 2).
//
// With many queries the key pool is re-read by every query, so the scan is a
// dense contraction and goes to tcgen05. A tile is QB = 256 / H_I queries of
// one sequence against 128 consecutive keys, computed transposed:
//   S^T [128 keys x 256 (query, head)] = K [128 x 128] . (Q^I)^T
// (M = 128, N = 256, K = 128, bf16 in, fp32 accumulate in tensor memory).
// A thread owns one key (one TMEM lane) and finds the H_I heads of a query in
// consecutive columns, so the ReLU-weighted head sum needs no exchange and a
// warp's stores of one query's scores are coalesced.
//
// Work: the tiles whose keys some query of the block can see. Every CTA
// counts them per query block from n_vis, then takes an equal contiguous range
// of the list (consecutive tiles share the query block, whose Q^I stays in
// shared memory). Keys are double-buffered with cp.async, and the two halves
// of tensor memory alternate so that the MMA of tile i overlaps the epilogue
// of tile i-1. A query block whose queries are not all of one valid sequence
// is scored with plain fp32 dot products instead.
#include "launchers.cuh"

namespace csa2 {

constexpr int kTcThreads = 256;  // 8 warps: warp w reads TMEM lanes 32(w%4).., column half w/4
constexpr int kTcKeys = 128;                       // keys per tile (M)
constexpr int kTcCols = 256;                       // (query, head) columns per tile (N)
constexpr int kTcMaxBlocks = 4096;                 // query blocks handled by the tensor-core form
constexpr uint32_t TC_Q = 0;                       // [2 dim blocks][256 rows][128 B]
constexpr uint32_t TC_K = TC_Q + 65536;            // [2 buffers][2 dim blocks][128 rows][128 B]
constexpr uint32_t TC_W = TC_K + 65536;            // [2 slots][256] head weights (query-major)
constexpr uint32_t TC_NV = TC_W + 2048;            // [2 slots][32] visible counts
constexpr uint32_t TC_CNT = TC_NV + 256;           // [kTcMaxBlocks] live tiles per query block
constexpr uint32_t TC_START = TC_CNT + 4 * kTcMaxBlocks;          // [kTcMaxBlocks + 1] their prefix
constexpr uint32_t TC_SCAL = TC_START + 4 * (kTcMaxBlocks + 4);   // [kTcMaxBlocks] 1: scalar block
constexpr uint32_t TC_MISC = TC_SCAL + kTcMaxBlocks;              // 2 mbarriers, tmem slot, scan scratch
constexpr uint32_t TC_TOTAL = TC_MISC + 128;
constexpr uint32_t kTcSmem = TC_TOTAL + 1024;      // + alignment slack
constexpr uint32_t kIdescIdx = idesc_bf16(128, 256, 0, 0);

struct IndexTcParams {
  int n_query, n_seq, heads;
  int64_t max_vis, ld;
  const uint16_t* q_idx;
  const float* w_heads;
  const uint16_t* keys;
  const int64_t* pool_off;
  const int32_t* seq_of_q;
  const int32_t* n_vis;
  float* scores;
  uint32_t* flags;
};

// visible keys of query q, clamped to its pool (flagging overreach); -1 for a bad query
__device__ __forceinline__ int tc_query_nv(const IndexTcParams& p, int q, bool report, int* seq, int64_t* row0) {
  const int b = p.seq_of_q[q];
  if (b < 0 || b >= p.n_seq) {
    if (report) set_flag(p.flags, CSA2_FLAG_BAD_QUERY);
    return -1;
  }
  int nv = p.n_vis[q];
  const int64_t plen = p.pool_off[b + 1] - p.pool_off[b];
  if (nv > plen || nv > p.max_vis) {
    if (report) set_flag(p.flags, CSA2_FLAG_NVIS_TOO_LARGE);
    nv = (int)min(plen, p.max_vis);
  }
  *seq = b;
  *row0 = p.pool_off[b];
  return max(nv, 0);
}

// Scores of query block qb on the CUDA cores (its queries are not all of one
// valid sequence): plain fp32 dot products of the exact bf16 values.
template <int HI>
__device__ void tc_block_scalar(const IndexTcParams& p, int qb) {
  constexpr int QB = kTcCols / HI;
  for (int ql = 0; ql < QB; ++ql) {
    const int q = qb * QB + ql;
    if (q >= p.n_query) break;
    int b;
    int64_t row0;
    const int nv = tc_query_nv(p, q, threadIdx.x == 0, &b, &row0);
    for (int j = threadIdx.x; j < nv; j += kTcThreads) {
      const uint16_t* kr = p.keys + (row0 + j) * kIdxDim;
      float s = 0.f;
      for (int h = 0; h < HI; ++h) {
        const uint16_t* qh = p.q_idx + ((int64_t)q * HI + h) * kIdxDim;
        float d = 0.f;
        for (int c = 0; c < kIdxDim; ++c)
          d = fmaf(__uint_as_float((uint32_t)qh[c] << 16), __uint_as_float((uint32_t)kr[c] << 16), d);
        s = fmaf(p.w_heads[(int64_t)q * HI + h], fmaxf(d, 0.f), s);
      }
      p.scores[(int64_t)q * p.ld + j] = s;
    }
  }
}

template <int HI>
__global__ void __launch_bounds__(kTcThreads, 1) index_score_tc_kernel(const IndexTcParams p) {
  constexpr int QB = kTcCols / HI;  // queries per block: 32, 16 or 8
  extern __shared__ uint8_t tc_smem_raw[];
  const uint32_t raw_s = smem_u32(tc_smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* sm = tc_smem_raw + (base_s - raw_s);
  float* wsm = reinterpret_cast<float*>(sm + TC_W);     // [2 slots][256]
  int* nvsm = reinterpret_cast<int*>(sm + TC_NV);       // [2 slots][32]
  int* cnt = reinterpret_cast<int*>(sm + TC_CNT);       // [n_qb]
  int* start = reinterpret_cast<int*>(sm + TC_START);   // [n_qb + 1]
  uint8_t* scal = sm + TC_SCAL;                         // [n_qb]
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + TC_MISC);  // [0..3] mbarriers, [4] tmem address
  int* scan_s = reinterpret_cast<int*>(sm + TC_MISC + 32);     // [4] warp totals
  const uint32_t mbar0 = base_s + TC_MISC;              // MMA into tensor-memory half 0 / 1 done
  const uint32_t tslot = base_s + TC_MISC + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_qb = (p.n_query + QB - 1) / QB;

  if (warp == 0) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(mbar0, 1);
    mbar_init(mbar0 + 8, 1);
    fence_mbar_init();
  }
  // ---- live tiles per query block: the key blocks below the block's largest
  // n_vis; a block not all of one valid sequence is one pseudo tile (scalar).
  // Lane l of a warp reads query base + l; groups of QB lanes form a block.
  for (int q0 = warp * 32; q0 < n_qb * QB; q0 += 32 * (kTcThreads / 32)) {
    const int q = q0 + lane;
    int nv = 0, sq = -1;
    if (q < p.n_query) {
      nv = (int)min((int64_t)max(p.n_vis[q], 0), p.max_vis);
      sq = p.seq_of_q[q];
      if (sq < 0 || sq >= p.n_seq) sq = -1;
    } else {
      sq = -3;  // past the end: neutral for the sequence test
    }
    int mx = nv, smin = sq == -3 ? 0x7FFFFFFF : sq, smax = sq == -3 ? -0x7FFFFFFF : sq;
    bool bad = sq == -1;
#pragma unroll
    for (int o = 1; o < QB; o <<= 1) {
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      smin = min(smin, __shfl_xor_sync(0xffffffffu, smin, o));
      smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, o));
      bad = __shfl_xor_sync(0xffffffffu, (int)bad, o) != 0 || bad;
    }
    const int qb = q / QB;
    if ((lane % QB) == 0 && qb < n_qb) {
      const bool homo = !bad && smin == smax;
      cnt[qb] = homo ? (mx + kTcKeys - 1) / kTcKeys : 1;
      scal[qb] = homo ? 0 : 1;
    }
  }
  __syncthreads();
  // ---- prefix of the live-tile counts: thread t sums a contiguous segment
  {
    const int per = (n_qb + kTcThreads - 1) / kTcThreads;
    const int i0 = min(n_qb, tid * per), i1 = min(n_qb, i0 + per);
    int lsum = 0;
    for (int i = i0; i < i1; ++i) lsum += cnt[i];
    int incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) scan_s[warp] = incl;
    __syncthreads();
    int run = incl - lsum;
    for (int w = 0; w < warp; ++w) run += scan_s[w];
    for (int i = i0; i < i1; ++i) {
      start[i] = run;
      run += cnt[i];
    }
    if (tid == kTcThreads - 1) start[n_qb] = run;
  }
  __syncthreads();
  const int total = start[n_qb];
  // this CTA's tiles: [t_begin, t_end) of the list (query block major)
  const int t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  const uint32_t taddr = misc[4];  // written by tcgen05.alloc (slot at TC_MISC + 16)
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  uint32_t mph[2] = {0u, 0u};
  bool aborted = false;

  // query block holding list position t (binary search over start)
  auto block_of = [&](int t) -> int {
    int lo = 0, hi = n_qb;  // start[lo] <= t < start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (start[mid] <= t) lo = mid;
      else hi = mid;
    }
    return lo;
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- the current query block: Q^I (cp.async, swizzled K-major rows
  // (query, head)), head weights and clamped visible counts
  int cur_qb = -1, qnvmax = 0;
  int64_t qrow0 = 0;
  auto load_block = [&](int b) {
    const int q0 = b * QB;
#pragma unroll 4
    for (int c = 0; c < (kTcCols * 16) / kTcThreads; ++c) {
      const int idx = tid + kTcThreads * c;
      const int row = idx >> 4, chunk = idx & 15;
      const bool ok = q0 + row / HI < p.n_query;
      const uint16_t* src = p.q_idx + ((int64_t)q0 * HI + row) * kIdxDim + 8 * chunk;
      const uint32_t dst = base_s + TC_Q + (uint32_t)(chunk >> 3) * 32768u + (uint32_t)row * 128u +
                           ((uint32_t)((chunk & 7) ^ (row & 7)) << 4);
      cp_async16(dst, ok ? src : p.q_idx, ok ? 16u : 0u);
    }
    for (int i = tid; i < kTcCols; i += kTcThreads)
      wsm[i] = (q0 + i / HI < p.n_query) ? p.w_heads[(int64_t)q0 * HI + i] : 0.f;
    if (tid < QB) {
      int nv = 0;
      if (q0 + tid < p.n_query) {
        int sq;
        int64_t r0;
        nv = max(0, tc_query_nv(p, q0 + tid, true, &sq, &r0));
      }
      nvsm[tid] = nv;
    }
    __syncthreads();
    qnvmax = 0;
    for (int i = 0; i < QB; ++i) qnvmax = max(qnvmax, nvsm[i]);
    qrow0 = p.pool_off[p.seq_of_q[q0]];
    cur_qb = b;
  };
  // keys kb*128 .. +127 of the current block's sequence into key buffer d
  auto load_keys = [&](int kb, int d) {
#pragma unroll 4
    for (int c = 0; c < (kTcKeys * 16) / kTcThreads; ++c) {
      const int idx = tid + kTcThreads * c;
      const int row = idx >> 4, chunk = idx & 15;
      const int64_t j = (int64_t)kb * kTcKeys + row;
      const bool ok = j < qnvmax;
      const uint16_t* src = p.keys + (qrow0 + j) * kIdxDim + 8 * chunk;
      const uint32_t dst = base_s + TC_K + (uint32_t)d * 32768u + (uint32_t)(chunk >> 3) * 16384u +
                           (uint32_t)row * 128u + ((uint32_t)((chunk & 7) ^ (row & 7)) << 4);
      cp_async16(dst, ok ? src : p.keys, ok ? 16u : 0u);
    }
  };
  // the MMA into tensor-memory half d has completed (its key buffer is free)
  auto epi_wait = [&](int d) -> bool {
    const bool ok = mbar_wait(mbar0 + 8u * (uint32_t)d, mph[d], p.flags);
    mph[d] ^= 1u;
    if (!__syncthreads_and(ok)) return false;
    tc_fence_after();
    return true;
  };
  // S^T of tile (block, kb) in tensor-memory half d -> scores: the thread
  // owns key row tid % 128 and column chunks 4 (tid / 128) .. +3
  auto epi_store = [&](int b, int kb, int d) {
    const int row = tid & (kTcKeys - 1), half = tid / kTcKeys;
    const int64_t j = (int64_t)kb * kTcKeys + row;
    const int q0 = b * QB;
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      const int c0 = 4 * half + 2 * cc;  // two 32-column chunks per round
      uint32_t r0[32], r1[32];
      tmem_ld32(taddr + (uint32_t)(256 * d + 32 * c0) + lane_base, r0);
      tmem_ld32(taddr + (uint32_t)(256 * d + 32 * c0 + 32) + lane_base, r1);
      float wc[64];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float4 v = reinterpret_cast<const float4*>(wsm + 32 * c0)[k];
        wc[4 * k] = v.x;
        wc[4 * k + 1] = v.y;
        wc[4 * k + 2] = v.z;
        wc[4 * k + 3] = v.w;
      }
      int nvc[64 / HI];
#pragma unroll
      for (int k = 0; k < 64 / HI; ++k) nvc[k] = nvsm[c0 * (32 / HI) + k];
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 64 / HI; ++k) {
        float sc = 0.f;
#pragma unroll
        for (int h = 0; h < HI; ++h) {
          const int col = k * HI + h;
          const float v = __uint_as_float(col < 32 ? r0[col] : r1[col - 32]);
          sc = fmaf(wc[col], fmaxf(v, 0.f), sc);
        }
        if (j < nvc[k]) p.scores[(int64_t)(q0 + c0 * (32 / HI) + k) * p.ld + j] = sc;
      }
    }
    tc_fence_before();
  };
  auto epilogue = [&](int b, int kb, int d) -> bool {
    if (!epi_wait(d)) return false;
    epi_store(b, kb, d);
    return true;
  };

  // ---- the tiles: MMA of tile i overlaps the epilogue of tile i-1, and the
  // keys of tile i+1 load meanwhile
  bool pend = false;
  int pend_b = 0, pend_kb = 0, pend_d = 0;
  int cur_d = 0;
  bool keys_ready = false;
  int b = t_begin < t_end ? block_of(t_begin) : 0;
  for (int t = t_begin; t < t_end && !aborted; ++t) {
    while (t >= start[b + 1]) ++b;
    const int kb = t - start[b];
    if (scal[b]) {
      if (pend) {
        aborted = !epilogue(pend_b, pend_kb, pend_d);
        pend = false;
      }
      __syncthreads();
      tc_block_scalar<HI>(p, b);
      keys_ready = false;
      continue;
    }
    if (b != cur_qb) {
      if (pend) {  // the last MMA that reads Q^I has to finish first
        aborted = !epilogue(pend_b, pend_kb, pend_d);
        pend = false;
        if (aborted) break;
      }
      __syncthreads();
      load_block(b);
      keys_ready = false;
    }
    if (!keys_ready) load_keys(kb, cur_d);
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      const uint32_t kbuf = base_s + TC_K + (uint32_t)cur_d * 32768u;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (uint32_t)(ks & 3) * 32u, kblk = (uint32_t)(ks >> 2);
        const uint64_t ad = sdesc_sw128(kbuf + kblk * 16384u + koff, 16u, 1024u);
        const uint64_t bd = sdesc_sw128(base_s + TC_Q + kblk * 32768u + koff, 16u, 1024u);
        mma_bf16_ss(taddr + 256u * (uint32_t)cur_d, ad, bd, kIdescIdx, ks > 0 ? 1u : 0u);
      }
      mma_commit(mbar0 + 8u * (uint32_t)cur_d);
    }
    // tile i-1's MMA done -> its key buffer takes the keys of tile i+1 (same
    // block), which load while tile i-1's scores are written
    if (pend) aborted = !epi_wait(pend_d);
    keys_ready = false;
    if (!aborted && t + 1 < t_end && t + 1 < start[b + 1]) {
      load_keys(kb + 1, cur_d ^ 1);
      keys_ready = true;
    }
    if (pend && !aborted) epi_store(pend_b, pend_kb, pend_d);
    pend = false;
    pend = true;
    pend_b = b;
    pend_kb = kb;
    pend_d = cur_d;
    cur_d ^= 1;
  }
  if (pend && !aborted) aborted = !epilogue(pend_b, pend_kb, pend_d);
  if (aborted) {
    // let tensor-core work still in flight land before its memory is freed
    mbar_wait(mbar0, mph[0], p.flags, 1000000000ull);
    mbar_wait(mbar0 + 8, mph[1], p.flags, 1000000000ull);
  }
  cp_async_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, 512);
}

bool index_tc_suited(int idx_fp8, int n_query, int n_seq, int idx_heads) {
  // many queries per sequence (chunked prefill): every key is read by many
  // queries, so the scan is a dense contraction
  return !idx_fp8 && (idx_heads == 8 || idx_heads == 16 || idx_heads == 32) && n_query >= 256 &&
         n_query >= 32 * n_seq && (n_query + kTcCols / idx_heads - 1) / (kTcCols / idx_heads) <= kTcMaxBlocks;
}

cudaError_t launch_index_score_tc(cudaStream_t st, int num_sms, int idx_heads, int n_query, int n_seq,
                                  int64_t max_vis, const uint16_t* q_idx, const float* w_heads, const uint16_t* keys,
                                  const int64_t* pool_off, const int32_t* seq_of_q, const int32_t* n_vis,
                                  float* scores, int64_t ld, uint32_t* flags) {
  if (n_query == 0 || max_vis == 0) return cudaSuccess;
  IndexTcParams p;
  p.n_query = n_query;
  p.n_seq = n_seq;
  p.heads = idx_heads;
  p.max_vis = max_vis;
  p.ld = ld;
  p.q_idx = q_idx;
  p.w_heads = w_heads;
  p.keys = keys;
  p.pool_off = pool_off;
  p.seq_of_q = seq_of_q;
  p.n_vis = n_vis;
  p.scores = scores;
  p.flags = flags;
  cudaError_t e = cudaSuccess;
  const dim3 grid((unsigned)num_sms);
#define CSA2_IDX_TC(HI)                                                                                     \
  do {                                                                                                    \
    e = cudaFuncSetAttribute(index_score_tc_kernel<HI>, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                             (int)kTcSmem);                                                              \
    if (e == cudaSuccess) index_score_tc_kernel<HI><<<grid, kTcThreads, kTcSmem, st>>>(p);                \
  } while (0)
  switch (idx_heads) {
    case 8: CSA2_IDX_TC(8); break;
    case 16: CSA2_IDX_TC(16); break;
    case 32: CSA2_IDX_TC(32); break;
    default: return cudaErrorInvalidValue;
  }
#undef CSA2_IDX_TC
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace csa2
