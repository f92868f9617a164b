// Pieces of the attention kernel of k_attend.cu (rows gathered, and
// converted from fp8 or fp4 where stored so, by the CTA's own threads): the
// shared-memory layout, the per-tile softmax and the output epilogue. They
// follow "Reading Notes of DeepSeek-V4.1-Flash", section 3a (softmax with
// the per-head sink in the denominator) and section 3f, C2 step 3 (the
// window plus the selected entries); "DeepSeek-V4.1-Flash on WASTE", "What
// is new" item 1 (the output's rope channels rotated back by -t).
//
// Per tile, in transposed form so that the 128 gathered rows are M = 128:
//   S^T [128 rows x 64 heads] = KV [128 x 512] . Q^T          (K = 512)
//   O^T [512 dims x 64 heads] += KV^T [512 x 128] . P^T       (K = 128)
// KV sits in shared memory once, in the 128-byte-swizzled layout that is at
// the same time the K-major A operand of the first product and the MN-major
// A operand of the second. S^T (64 columns) and O^T (4 x 64 columns) live in
// tensor memory. Softmax runs with one thread per (row = TMEM lane, half of
// the heads): warp w reads lane quadrant w % 4 and heads 32 (w / 4) .. +31.
#pragma once
#include "launchers.cuh"

namespace csa2 {

constexpr int kTileRows = 128;
// 8 math warps: warp w reads tensor-memory lane quadrant w % 4 (tile rows, or
// output dims, 32 (w % 4) .. +31) and takes heads 32 (w / 4) .. +31 of them
constexpr int kAttWarps = 8;
constexpr int kAttThreads = 32 * kAttWarps;
constexpr int kKvGroups = 4;  // bf16 tiles land in 4 groups of two 64-channel blocks
constexpr uint32_t SM_Q = 0;                          // [9 dim blocks][64 heads][128 B]; block 8 = rope residual
constexpr uint32_t SM_KV = 73728;                     // [8 dim blocks][128 rows][128 B]
constexpr uint32_t SM_P = SM_KV + 131072;             // [128 rows][128 B]  (64 heads, bf16)
constexpr uint32_t SM_RED = SM_P + 16384;             // float [4][64]
constexpr uint32_t SM_MRUN = SM_RED + 1024;           // float [64]
constexpr uint32_t SM_LRUN = SM_MRUN + 256;           // float [64]
constexpr uint32_t SM_MUSE = SM_LRUN + 256;           // float [64]
constexpr uint32_t SM_ALPHA = SM_MUSE + 256;          // float [64]
constexpr uint32_t SM_ROWS = SM_ALPHA + 256;          // int64 [128] row sources (thread-gathered kernel)
constexpr uint32_t SM_MISC = SM_ROWS + 1024;          // mbarrier, tmem slot, flags
constexpr uint32_t SM_ROPE = SM_MISC + 64;            // float2 [32]: cos, sin of t * f_i
constexpr uint32_t SM_TOTAL = SM_ROPE + 256;
constexpr uint32_t kAttSmemBytes = SM_TOTAL + 1024;   // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescQK = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, 1, 1);

// Butterfly reduce-scatter of 32 per-lane values over the 32 lanes of a warp:
// afterwards lane l holds the reduction of value l (step k exchanges the
// half that lane bit 4-k selects).
template <bool MAX>
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 16 >> step;
    const int off = 16 >> step;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < half) {
        const float lo = v[i], hi = v[half + i];
        const float send = upper ? lo : hi;
        const float keep = upper ? hi : lo;
        const float recv = __shfl_xor_sync(0xffffffffu, send, off);
        v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
      }
    }
  }
  return v[0];
}

// Barriers of the CTA's 256 threads, passed to the shared pieces below.
struct SyncCta {
  __device__ __forceinline__ void sync() const { __syncthreads(); }
  __device__ __forceinline__ bool any(bool v) const { return __syncthreads_or(v) != 0; }
  __device__ __forceinline__ bool all(bool v) const { return __syncthreads_and(v) != 0; }
};

// Where one query's rows live: its position t, the first window position it
// sees (lo_eff), its sequence's window buffer and pool.
struct QueryRows {
  int64_t t, lo_eff, win_b0, win_cap, pool_b0, plen;
};

__device__ __forceinline__ QueryRows query_rows(const AttendParams& p, int64_t t, int bs, bool q_ok) {
  QueryRows qr;
  qr.t = t;
  qr.win_b0 = p.win_off[bs];
  qr.win_cap = q_ok ? (p.win_off[bs + 1] - qr.win_b0) : 0;
  // no selection (window-only call): the pool arguments may be NULL
  qr.pool_b0 = p.pool_off != nullptr ? p.pool_off[bs] : 0;
  qr.plen = (q_ok && p.pool_off != nullptr) ? (p.pool_off[bs + 1] - qr.pool_b0) : 0;
  const int64_t lo_raw = (q_ok && p.win_lo) ? p.win_lo[bs] : 0;
  qr.lo_eff = max(max((int64_t)0, lo_raw), t - (int64_t)p.window + 1);
  return qr;
}

// Source row of row r of a query's tile (tile 0: window position lo_eff + r;
// selected tile: entry j of the selection), -1 for none; bad values are
// recorded in the error word and skipped.
__device__ __forceinline__ int64_t tile_row_src(const AttendParams& p, const QueryRows& qr, int tile, int r,
                                                int32_t j) {
  int64_t src = -1;
  if (tile == 0) {
    const int64_t pos = qr.lo_eff + r;
    if (pos <= qr.t && r < p.window) {
      if (qr.t - qr.lo_eff + 1 > qr.win_cap) set_flag(p.flags, CSA2_FLAG_BAD_WINDOW);
      else src = qr.win_b0 + (pos % qr.win_cap);
    }
  } else if (j >= 0 && j >= p.shard_lo && j < p.shard_hi) {
    // entries outside this launch's shard of the pool are not its rows
    const int64_t jr = (int64_t)j - p.shard_lo;
    if (jr < qr.plen) src = qr.pool_b0 + jr;
    else set_flag(p.flags, CSA2_FLAG_BAD_TOPK_INDEX);
  } else if (j < -1) {
    set_flag(p.flags, CSA2_FLAG_BAD_TOPK_INDEX);
  }
  return src;
}

// Q of query qi copied asynchronously into its swizzled K-major slots (dim
// blocks 0..7), by the 256 threads; the caller commits the group.
__device__ __forceinline__ void copy_q_async(const AttendParams& p, uint32_t base_s, int qi) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int h = warp; h < kHeads; h += kAttWarps) {
    const uint16_t* qh = p.q + ((int64_t)qi * kHeads + h) * kDim;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = lane + 32 * cc;  // 16-byte chunk: channels 8c .. 8c+7
      const uint32_t dst = base_s + SM_Q + (uint32_t)(c >> 3) * 8192u + (uint32_t)h * 128u +
                           ((uint32_t)((c & 7) ^ (h & 7)) << 4);
      cp_async16(dst, qh + 8 * c, 16u);
    }
  }
}

// bf16 rows of a tile gathered asynchronously into the swizzled KV operand
// in kKvGroups commit groups, one per pair of 64-channel blocks (a half warp
// copies one row's 256 B of a pair); a missing row (-1) reads zeros.
__device__ __forceinline__ void gather_bf16_tile(uint32_t base_s, const int64_t* rows, const uint16_t* kv) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int g = 0; g < kKvGroups; ++g) {
#pragma unroll
    for (int u = 0; u < kTileRows * 16 / kAttThreads; ++u) {
      const int i = tid + kAttThreads * u;
      const int r = i >> 4;
      const int c = 16 * g + (i & 15);
      const int64_t src = rows[r];
      const uint32_t dst = base_s + SM_KV + (uint32_t)(c >> 3) * 16384u + (uint32_t)r * 128u +
                           ((uint32_t)((c & 7) ^ (r & 7)) << 4);
      const uint16_t* gp = src >= 0 ? kv + src * kDim + 8 * c : kv;
      cp_async16(dst, gp, src >= 0 ? 16u : 0u);
    }
    cp_async_commit();
  }
}

// S^T = KV . Q^T, the K steps of channel-block group g of n_groups (steps
// 0..31 cover the 8 channel blocks; with the rope residual, the last group
// adds steps 32..35: q's residual block against the KV's last channel
// block). Descriptors are constant offsets from the operands' bases: one
// issuing thread, not the tensor pipe, bounds these N = 64 products.
// Called by one thread.
__device__ __forceinline__ void issue_qk(uint32_t base_s, uint32_t tmem_s, int g, int n_groups, bool rope) {
  const uint64_t ad0 = sdesc_sw128(base_s + SM_KV, 16u, 1024u);
  const uint64_t bd0 = sdesc_sw128(base_s + SM_Q, 16u, 1024u);
  const int ks0 = g * 32 / n_groups, ks1 = (g + 1) * 32 / n_groups;
#pragma unroll
  for (int ks = ks0; ks < ks1; ++ks)
    mma_bf16_ss(tmem_s, sdesc_add(ad0, (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u),
                sdesc_add(bd0, (uint32_t)(ks >> 2) * 8192u + (uint32_t)(ks & 3) * 32u), kIdescQK, ks > 0 ? 1u : 0u);
  if (g == n_groups - 1 && rope) {
#pragma unroll
    for (int ks = 32; ks < 36; ++ks)
      mma_bf16_ss(tmem_s, sdesc_add(ad0, 7u * 16384u + (uint32_t)(ks & 3) * 32u),
                  sdesc_add(bd0, 8u * 8192u + (uint32_t)(ks & 3) * 32u), kIdescQK, 1u);
  }
}

// O^T (+)= KV^T . P^T in four blocks of 128 output dims (accumulate: add to
// what O^T holds). Called by one thread.
__device__ __forceinline__ void issue_pv(uint32_t base_s, uint32_t tmem_o, bool accumulate) {
  const uint64_t ad0 = sdesc_sw128(base_s + SM_KV, 16384u, 1024u);
  const uint64_t bd0 = sdesc_sw128(base_s + SM_P, 8192u, 1024u);
  const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_bf16_ss(tmem_o + 64u * (uint32_t)mt, sdesc_add(ad0, (uint32_t)(2 * mt) * 16384u + (uint32_t)ks * 2048u),
                  sdesc_add(bd0, (uint32_t)ks * 2048u), kIdescPV, ks > 0 ? 1u : acc0);
  }
}

// q's rope channels rotated in place, as hi + lo (both bf16) in dim block 7
// and the residual block 8: the tensor cores then see the rotation to ~2^-16
// relative instead of one bf16 rounding. Thread: head tid/4, chunks
// 56 + 2*(tid&3) .. +1 (the last 64 channels). Called by the 256 math
// threads once Q has landed.
__device__ __forceinline__ void q_rope_split(uint8_t* sm, const RopeParams& rp) {
  const int tid = threadIdx.x;
  const float2* rope_tab = reinterpret_cast<const float2*>(sm + SM_ROPE);
  const int h = tid >> 2;
  const int first_rope = kDim - 2 * rp.pairs;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int c = 56 + 2 * (tid & 3) + u;
    const uint32_t inblk = (uint32_t)h * 128u + ((uint32_t)((c & 7) ^ (h & 7)) << 4);
    uint4* hi_p = reinterpret_cast<uint4*>(sm + SM_Q + 7u * 8192u + inblk);
    const uint4 v = *hi_p;
    uint32_t w[4] = {v.x, v.y, v.z, v.w}, lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 cs2 = rope_tab[(8 * c + 2 * k - first_rope) >> 1];
      const float x0 = bf16lo(w[k]), x1 = bf16hi(w[k]);
      const float y0 = x0 * cs2.x - x1 * cs2.y, y1 = x0 * cs2.y + x1 * cs2.x;
      w[k] = pack_bf16(y0, y1);
      lo[k] = pack_bf16(y0 - bf16lo(w[k]), y1 - bf16hi(w[k]));
    }
    *hi_p = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(sm + SM_Q + 8u * 8192u + inblk) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Softmax over one tile's rows, after S^T has landed in tensor memory
// (thread = row = TMEM lane; heads 32 hh .. +31 of warp w, hh = w / 4).
// A head's reference max moves only when a tile exceeds it by more than 2^8:
// P = 2^(s - m) then stays below 256 and the softmax is the same for any
// reference, so most tiles skip both the max reduction (a vote checks the
// bound) and the O^T rescale. Writes P^T (bf16, the MN-major B operand of the
// PV product), adds the bf16-rounded weights to this thread's unreduced row
// sums lsum (scaled with the reference when it moves), rescales O^T in
// tensor memory where needed, and ends with the async-proxy fence and a
// barrier of the math threads: P^T and O^T are then ready for the PV product.
template <class Sync>
__device__ __forceinline__ void tile_softmax(const AttendParams& p, uint8_t* sm, uint32_t tmem_s, uint32_t tmem_o,
                                             uint32_t lane_base, bool valid, bool first, uint32_t* rescale,
                                             float (&lsum)[32], const Sync& sy) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, hh = warp >> 2;
  const int row = quad * 32 + lane;
  float* red = reinterpret_cast<float*>(sm + SM_RED);
  float* m_run = reinterpret_cast<float*>(sm + SM_MRUN);
  float* m_use = reinterpret_cast<float*>(sm + SM_MUSE);
  float* alpha = reinterpret_cast<float*>(sm + SM_ALPHA);
  float s[32];
  {
    uint32_t r0[32];
    tmem_ld32(tmem_s + lane_base + 32 * hh, r0);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 32; ++k) s[k] = valid ? __uint_as_float(r0[k]) * p.scale_log2 : -INFINITY;
  }
  bool need_max = first;
  if (!need_max) {
    bool over = false;
#pragma unroll
    for (int k = 0; k < 32; ++k) over |= s[k] > m_run[32 * hh + k] + 8.f;
    need_max = sy.any(over);
  }
  if (need_max) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = s[k];
    red[quad * 64 + 32 * hh + lane] = reduce_scatter32<true>(v, lane);
  }
  sy.sync();
  if (!need_max) {
    if (tid < kHeads) alpha[tid] = 1.f;  // m_use and m_run stand
  } else if (tid < kHeads) {
    const float tmax = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
    const float mo = m_run[tid];
    const float mn = (mo == -INFINITY || tmax > mo + 8.f) ? fmaxf(mo, tmax) : mo;
    const float mu = (mn == -INFINITY) ? 0.f : mn;
    const float al = (mo == -INFINITY) ? 1.f : exp2f(mo - mu);
    m_use[tid] = mu;
    alpha[tid] = al;
    m_run[tid] = mn;
    if (al != 1.f && !first) *rescale = 1;
  }
  sy.sync();
  const bool do_rescale = *rescale != 0;
  {
    if (do_rescale) {
#pragma unroll
      for (int k = 0; k < 32; ++k) lsum[k] *= alpha[32 * hh + k];
    }
    uint32_t packed[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float p0 = exp2f(s[2 * k] - m_use[32 * hh + 2 * k]);
      const float p1 = exp2f(s[2 * k + 1] - m_use[32 * hh + 2 * k + 1]);
      packed[k] = pack_bf16(p0, p1);
      lsum[2 * k] += bf16lo(packed[k]);  // the weights PV sums, rounded to bf16
      lsum[2 * k + 1] += bf16hi(packed[k]);
    }
    // P^T row `row`: 64 heads = 8 chunks of 16 B; this thread writes chunks
    // 4 hh .. 4 hh + 3
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const int c = 4 * hh + c4;
      const uint32_t off = SM_P + (uint32_t)row * 128u + ((uint32_t)(c ^ (row & 7)) << 4);
      *reinterpret_cast<uint4*>(sm + off) =
          make_uint4(packed[4 * c4], packed[4 * c4 + 1], packed[4 * c4 + 2], packed[4 * c4 + 3]);
    }
  }
  if (do_rescale) {
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
      uint32_t r[32];
      const uint32_t a = tmem_o + (uint32_t)(64 * mt + 32 * hh) + lane_base;
      tmem_ld32(a, r);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha[32 * hh + k]);
      tmem_st32(a, r);
    }
    tmem_wait_st();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  sy.sync();
  if (tid == 0) *rescale = 0;  // read by every thread before the barrier above
}

// One 128-dim block (dims 128 mt ..) of a [64 heads][512] bf16 output from
// the threads' fp32 values v (thread: dim 128 mt + row, heads 32 hh .. +31).
// Lanes d, d+1 swap halves so that each holds two adjacent dims of one head
// (the even lane head k, the odd lane head k+1), and the pairs are staged in
// the P buffer (free once the last PV product is done) as [head][128 dims],
// the 16-byte chunks of odd heads shifted by four so that the two halves of a
// warp write different banks. The block then leaves in coalesced 16-byte
// stores, 256 B per head.
template <class Sync>
__device__ __forceinline__ void store_out_block(uint8_t* sm, const float (&v)[32], int mt, uint16_t* dst,
                                                const Sync& sy) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, hh = warp >> 2;
  const int p2 = (quad * 32 + lane) >> 1;  // dim pair of this thread in the block
  const bool odd = (lane & 1) != 0;
  uint8_t* stage = sm + SM_P;
#pragma unroll
  for (int k = 0; k < 32; k += 2) {
    const float recv = __shfl_xor_sync(0xffffffffu, odd ? v[k] : v[k + 1], 1);
    const int h = 32 * hh + k + (odd ? 1 : 0);
    const uint32_t w = odd ? pack_bf16(recv, v[k + 1]) : pack_bf16(v[k], recv);
    const int chunk = (p2 >> 2) ^ ((h & 1) << 2);
    *reinterpret_cast<uint32_t*>(stage + h * 256 + chunk * 16 + (p2 & 3) * 4) = w;
  }
  sy.sync();
#pragma unroll
  for (int u = 0; u < kHeads * 16 / kAttThreads; ++u) {
    const int c = tid + kAttThreads * u;
    const int h = c >> 4, part = c & 15;
    const uint4 x = *reinterpret_cast<const uint4*>(stage + h * 256 + ((part ^ ((h & 1) << 2)) * 16));
    *reinterpret_cast<uint4*>(dst + (int64_t)h * kDim + 128 * mt + 8 * part) = x;
  }
  sy.sync();  // the stage is free for the next block
}

// The epilogue of a CTA's tiles, by the 256 math threads once the last PV
// product has completed: the row sums reduced, then one of
//   direct == 2: the unnormalised partial (O^T, m in natural-log units, l) of
//                csa2_attend_partial, no sink, no rotation back;
//   direct == 1: the output normalised with the sink, rope channels rotated
//                back by -t, and lse;
//   direct == 0: the bf16 partial and (m, l) of this split for the merge.
template <class Sync>
__device__ __forceinline__ void attend_store(const AttendParams& p, uint8_t* sm, int qi, int split, bool have_o,
                                             float (&lsum)[32], uint32_t tmem_o, uint32_t lane_base, float sink_l2,
                                             const Sync& sy) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, hh = warp >> 2;
  const int row = quad * 32 + lane;
  float* red = reinterpret_cast<float*>(sm + SM_RED);
  float* m_run = reinterpret_cast<float*>(sm + SM_MRUN);
  float* l_run = reinterpret_cast<float*>(sm + SM_LRUN);
  float* alpha = reinterpret_cast<float*>(sm + SM_ALPHA);
  const float2* rope_tab = reinterpret_cast<const float2*>(sm + SM_ROPE);
  if (have_o) {
    // the row sums: over this warp's 32 rows (lanes), then over the 4 quadrants
    red[quad * 64 + 32 * hh + lane] = reduce_scatter32<false>(lsum, lane);
    sy.sync();
    if (tid < kHeads) l_run[tid] = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
    sy.sync();
  }
  const int first_rope = kDim - 2 * p.rp.pairs;
  if (p.direct == 2) {
    if (tid < kHeads) {
      const int64_t o = (int64_t)qi * kHeads + tid;
      p.part_m[o] = have_o ? m_run[tid] * 0.6931471805599453f : -INFINITY;
      p.part_l[o] = have_o ? l_run[tid] : 0.f;
    }
    float* po = p.part_o + (int64_t)qi * kHeads * kDim;
    for (int mt = 0; mt < 4; ++mt) {
      const int d = 128 * mt + row;
      uint32_t r[32];
      if (have_o) {
        tmem_ld32(tmem_o + (uint32_t)(64 * mt + 32 * hh) + lane_base, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) po[(int64_t)(32 * hh + k) * kDim + d] = __uint_as_float(r[k]);
    }
  } else if (p.direct) {
    // final normalisation with the sink: fo = e^{m - M} / den, den = l e^{m - M} + e^{sink - M}
    if (tid < kHeads) {
      const float sk = sink_l2;
      const float mr = have_o ? m_run[tid] : -INFINITY;
      const float M = fmaxf(mr, sk);
      float fo = 0.f, lse = -INFINITY;
      if (M != -INFINITY) {
        const float em = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
        const float den = l_run[tid] * em + exp2f(sk - M);
        fo = em / den;
        lse = (M + log2f(den)) * 0.6931471805599453f;
      }
      alpha[tid] = fo;
      if (p.lse) p.lse[(int64_t)qi * kHeads + tid] = lse;
    }
    sy.sync();
    uint16_t* out = p.out + (int64_t)qi * kHeads * kDim;
    float al_all[32];  // this warp's head half, before any store: no reloads
#pragma unroll
    for (int k = 0; k < 32; ++k) al_all[k] = alpha[32 * hh + k];
    for (int mt = 0; mt < 4; ++mt) {
      const int d = 128 * mt + row;
      uint32_t ra[32];
      if (have_o) {
        tmem_ld32(tmem_o + (uint32_t)(64 * mt + 32 * hh) + lane_base, ra);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) ra[k] = 0u;
      }
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(ra[k]) * al_all[k];
      // rope channels rotated back by -t: only warps that hold some exchange
      // values with the pair's other lane (warp-uniform test)
      if (p.rp.pairs > 0 && 128 * mt + 32 * quad + 31 >= first_rope) {
        const bool rope = d >= first_rope;
        float cs = 1.f, sn = 0.f;
        if (rope) {
          const float2 cs2 = rope_tab[(d - first_rope) >> 1];
          cs = cs2.x;
          sn = cs2.y;
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float partner = __shfl_xor_sync(0xffffffffu, v[k], 1);
          if (rope) v[k] = (d & 1) ? (v[k] * cs - partner * sn) : (v[k] * cs + partner * sn);
        }
      }
      store_out_block(sm, v, mt, out, sy);
    }
  } else {
    // unnormalised partial O^T and (m, l) for the merge
    const int64_t slot = (int64_t)qi * p.n_slots + p.slot_base + split;
    if (tid < kHeads)
      p.ws_ml[slot * kHeads + tid] = make_float2(have_o ? m_run[tid] : -INFINITY, have_o ? l_run[tid] : 0.f);
    if (have_o) {
      // bf16 partials: the merge's weighted sum then carries 2^-8 of each
      // partial's magnitude
      uint16_t* wo = p.ws_o + slot * kHeads * kDim;
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t r[32];
        tmem_ld32(tmem_o + (uint32_t)(64 * mt + 32 * hh) + lane_base, r);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
        store_out_block(sm, v, mt, wo, sy);
      }
    }
  }
}

}  // namespace csa2
