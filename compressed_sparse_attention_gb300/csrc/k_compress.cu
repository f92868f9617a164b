// Row storage (RoPE + bf16 / fp8-block-32 store) and the CSA2 compressor.
//
// Compressor: "Reading Notes of DeepSeek-V4.1-Flash", section 3f, C2 step 1
// (softmax-gated pooling of m consecutive tokens); "DeepSeek-V4.1-Flash on
// WASTE", "What is new" item 1 (fp32 pooling, then RMS-normalised); PocketLLM
// "DeepSeek-V4.1-Flash", "The CSA2 attention layers" (the index key is taken
// from the unrotated latent; the latent is rotated at its group's first token
// position j*m before it is stored).
#include "launchers.cuh"

namespace csa2 {

// ---------------------------------------------------------------------------
// store_rows: one warp per row; lane owns DIM/32 contiguous channels.
// ---------------------------------------------------------------------------
// FMT: 0 bf16, 1 fp8 (e4m3 + ue8m0 / 32), 2 fp4 (e2m1 + e4m3 / 16), 3 mxfp4 (e2m1 + ue8m0 / 32)
template <int DIM, int FMT>
__global__ void __launch_bounds__(256) store_rows_kernel(const float* __restrict__ rows, int64_t n_rows,
                                                         const int64_t* __restrict__ pos, RopeParams rp,
                                                         void* __restrict__ out, uint8_t* __restrict__ out_scale) {
  constexpr int E = DIM / 32;  // channels per lane (4 or 16)
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  float v[E];
  const float4* src = reinterpret_cast<const float4*>(rows + row * DIM + lane * E);
#pragma unroll
  for (int k = 0; k < E / 4; ++k) {
    float4 f = src[k];
    v[4 * k] = f.x; v[4 * k + 1] = f.y; v[4 * k + 2] = f.z; v[4 * k + 3] = f.w;
  }
  if (pos != nullptr && rp.pairs > 0) {
    const int64_t p = pos[row];
    const int first = DIM - 2 * rp.pairs;
#pragma unroll
    for (int k = 0; k < E; k += 2) {
      const int ch = lane * E + k;
      if (ch >= first) {
        float c, s;
        rope_cs(rp, (ch - first) >> 1, p, c, s);
        const float x0 = v[k], x1 = v[k + 1];
        v[k] = x0 * c - x1 * s;
        v[k + 1] = x0 * s + x1 * c;
      }
    }
  }
  if constexpr (FMT == 0) {
    uint32_t w[E / 2];
#pragma unroll
    for (int k = 0; k < E / 2; ++k) w[k] = pack_bf16(v[2 * k], v[2 * k + 1]);
    uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(out) + row * DIM + lane * E);
#pragma unroll
    for (int k = 0; k < E / 4; ++k) dst[k] = make_uint2(w[2 * k], w[2 * k + 1]);
  } else if constexpr (FMT == 1) {
    constexpr int LPB = 32 / E;  // lanes per 32-channel block
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(v[k]));
#pragma unroll
    for (int o = 1; o < LPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const uint32_t eb = fp8_scale_byte(amax);
    const int sh = 127 - (int)eb;  // x / 2^(eb-127), exact
    uint8_t* dst = reinterpret_cast<uint8_t*>(out) + row * DIM + lane * E;
#pragma unroll
    for (int k = 0; k < E; k += 4) {
      uint32_t word = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) word |= (uint32_t)f32_to_e4m3(ldexpf(v[k + u], sh)) << (8 * u);
      *reinterpret_cast<uint32_t*>(dst + k) = word;
    }
    if ((lane % LPB) == 0) out_scale[row * (DIM / 32) + lane / LPB] = (uint8_t)eb;
  } else {
    constexpr int BLK = (FMT == 2) ? 16 : 32;  // channels per scale
    constexpr int LPB = (BLK / E) > 0 ? BLK / E : 1;  // lanes per block
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(v[k]));
#pragma unroll
    for (int o = 1; o < LPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float sc;
    uint32_t sbyte;
    if constexpr (FMT == 2) {
      sbyte = fp4_scale_e4m3(amax);
      sc = e4m3_value(sbyte);
    } else {
      sbyte = mxfp4_scale_byte(amax);
      sc = ue8m0_value(sbyte);
    }
    uint8_t* dst = reinterpret_cast<uint8_t*>(out) + row * (DIM / 2) + lane * (E / 2);
#pragma unroll
    for (int k = 0; k < E; k += 2) dst[k / 2] = (uint8_t)(e2m1_code(v[k], sc) | (e2m1_code(v[k + 1], sc) << 4));
    if ((lane % LPB) == 0) out_scale[row * (DIM / BLK) + lane / LPB] = (uint8_t)sbyte;
  }
}

// ---------------------------------------------------------------------------
// compress: one CTA of 256 threads per closed group; thread t owns channels
// 2t, 2t+1 of the 512-wide latent. The kernel is latency-bound (a few KB per
// group), so every independent load is issued as early as possible: the
// index-key weights (warp w owns outputs 16w .. 16w+15, 32 x 16 B per lane)
// at kernel start, the segment lookup as a warp-parallel search.
// ---------------------------------------------------------------------------
constexpr int kCmpThreads = 256;

// largest b in [0, n) with off[b] <= x (off non-decreasing, off[0] = 0); warp-wide
__device__ __forceinline__ int find_segment_warp(const int64_t* __restrict__ off, int n, int64_t x) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int stride = (hi - lo + 31) / 32;
    const int i = lo + lane * stride;
    const bool le = i < hi && off[i] <= x;
    const int cnt = __popc(__ballot_sync(0xffffffffu, le));  // >= 1: off[lo] <= x
    const int nlo = lo + (cnt - 1) * stride;
    hi = min(hi, nlo + stride);
    lo = nlo;
  }
  return lo;
}

// Append form: sequence b closes g_b = floor((p_b + n_b) / m) - floor(p_b / m)
// groups (p_b its first new position, n_b its new tokens); CTA i takes the
// i-th closing group in sequence order. Warp-wide; false past the last one.
__device__ __forceinline__ bool find_append_group(const int64_t* __restrict__ tok_off,
                                                  const int64_t* __restrict__ first_pos, int n_seq, int m,
                                                  int64_t i, int* b_out, int64_t* j_out) {
  const int lane = threadIdx.x & 31;
  int64_t base = 0;
  for (int s0 = 0; s0 < n_seq; s0 += 32) {
    const int b = s0 + lane;
    int64_t g = 0;
    if (b < n_seq) {
      const int64_t p = first_pos[b], n = tok_off[b + 1] - tok_off[b];
      g = (p >= 0 && n >= 0) ? (p + n) / m - p / m : 0;
    }
    int64_t incl = g;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int64_t total = __shfl_sync(0xffffffffu, incl, 31);
    if (i < base + total) {
      const int64_t excl = base + incl - g;
      const unsigned bal = __ballot_sync(0xffffffffu, g > 0 && excl <= i && i < excl + g);
      const int src = __ffs(bal) - 1;
      const int64_t e = __shfl_sync(0xffffffffu, excl, src);
      *b_out = s0 + src;
      *j_out = first_pos[s0 + src] / m + (i - e);
      return true;
    }
    base += total;
  }
  return false;
}

// The index-key weights W^I [128][512] bf16 as the per-group code reads
// them: warp w takes rows 16w .. 16w+15, lane l channels 16l .. 16l+15 of
// each (a: the first 8, b: the last 8). A few groups (decode) hold them in
// registers (247 registers, one CTA per SM); their loads go out right after
// the group's own tokens, so that the tokens are not queued behind 128 KiB of
// weights. Many groups (chunked prefill) load them where they are used (98
// registers, two CTAs per SM, so that two groups' latency chains overlap on
// each SM): 2,048 groups take 44 µs instead of 69 µs. Both read the same
// values in the same order.
struct CmpWRegs {
  const uint16_t* w;
  uint4 wa[16], wb[16];
  __device__ __forceinline__ void load() {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const uint4* wr = reinterpret_cast<const uint4*>(w + (int64_t)(warp * 16 + u) * kDim + 16 * lane);
      wa[u] = wr[0];
      wb[u] = wr[1];
    }
  }
  __device__ __forceinline__ void get(int u, uint4& a, uint4& b) const {
    a = wa[u];
    b = wb[u];
  }
};
struct CmpWGlobal {
  const uint16_t* w;
  __device__ __forceinline__ void load() {}
  __device__ __forceinline__ void get(int u, uint4& a, uint4& b) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint4* wr = reinterpret_cast<const uint4*>(w + (int64_t)(warp * 16 + u) * kDim + 16 * lane);
    a = __ldg(wr);
    b = __ldg(wr + 1);
  }
};

struct CmpArgs {
  const uint16_t* raw;
  const float* gate;
  int m, n_seq;
  const int64_t* tok_off;
  const int64_t* first_pos;
  const int64_t* pool_off;
  int idx_dim;
  float eps;
  RopeParams rp;
  void* pool_kv;
  uint8_t* pool_kv_scale;
  void* idx_keys;
  uint8_t* idx_key_scale;
  uint32_t* flags;
  int append;
  const uint16_t* st_raw;
  const float* st_gate;
};

// One closed group grp (the whole-group form's group index, or the append
// form's running group number), by the CTA's 256 threads: pooling, norm,
// index key (when has_w), rope, store, and the tail scores. nw, knw: this
// thread's norm weights; w.load() issues the index-key weights' loads (a
// no-op where they are read in place). Every thread returns at the same point.
template <int KVF, int IKF, class W>
__device__ __forceinline__ void compress_group(const CmpArgs& A, int64_t grp, bool has_w, W& w, float2 nw, float knw,
                                               const CompressTail& tail) {
  __shared__ float c_hat_s[kDim];
  __shared__ float k_lin_s[kIdxDim];
  __shared__ float k_st_s[kIdxDim];  // the stored key's exact values (tail scoring)
  __shared__ float red_s[8];
  __shared__ int64_t seg_s[2];       // whole-group form: warp 0's segment lookup (j, pool row)
  __shared__ int segb_s[2];          // its sequence and a bad-segment mark
  __shared__ int tq_s[kCmpThreads];  // tail: the queries that score this entry
  __shared__ int tq_n;
  const uint16_t* __restrict__ raw = A.raw;
  const float* __restrict__ gate = A.gate;
  const int m = A.m, n_seq = A.n_seq;
  const int64_t* __restrict__ tok_off = A.tok_off;
  const int64_t* __restrict__ first_pos = A.first_pos;
  const int64_t* __restrict__ pool_off = A.pool_off;
  const int idx_dim = A.idx_dim;
  const float eps = A.eps;
  const RopeParams& rp = A.rp;
  void* __restrict__ pool_kv = A.pool_kv;
  uint8_t* __restrict__ pool_kv_scale = A.pool_kv_scale;
  void* __restrict__ idx_keys = A.idx_keys;
  uint8_t* __restrict__ idx_key_scale = A.idx_key_scale;
  uint32_t* flags = A.flags;
  const int append = A.append;
  const uint16_t* __restrict__ st_raw = A.st_raw;
  const float* __restrict__ st_gate = A.st_gate;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c0 = 2 * tid;
  uint32_t rw[16];
  float2 gv[16];
  int64_t j = 0, prow = 0;
  int seq_b = 0;
  // tail scoring: this thread's query (the first 256), its sequence and
  // visible length, loaded before anything depends on them
  const bool tail_on = has_w && tail.scores != nullptr;
  int sq = -1, nvq = 0;
  if (tid == 0) tq_n = 0;
  if (!append) {
    const int64_t tok0 = grp * m;
    // the group's tokens depend only on the group index: their loads go out
    // first (m <= 16); the pooling does not wait for the segment lookup
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (u < m) {
        rw[u] = *reinterpret_cast<const uint32_t*>(raw + (tok0 + u) * kDim + c0);
        gv[u] = m > 1 ? *reinterpret_cast<const float2*>(gate + (tok0 + u) * kDim + c0) : make_float2(0.f, 0.f);
      }
    }
    if (tail_on && tid < tail.n_query) {
      sq = tail.seq_of_q[tid];
      nvq = tail.n_vis[tid];
    }
    if (warp == 0) {  // the others go on to the weights; read back after the first barrier
      const int b = find_segment_warp(tok_off, n_seq, tok0);
      const int64_t seg0 = tok_off[b], seg1 = tok_off[b + 1], fp = first_pos[b];
      const int64_t pos0 = fp + (tok0 - seg0);  // position of the group's first token
      const int64_t jj = pos0 / m;
      const int64_t pr = pool_off[b] + jj;
      const bool bad = (seg0 % m) != 0 || ((seg1 - seg0) % m) != 0 || (fp % m) != 0 || fp < 0 || tok0 >= seg1 ||
                       pr >= pool_off[b + 1];
      if (lane == 0) {
        seg_s[0] = jj;
        seg_s[1] = pr;
        segb_s[0] = b;
        segb_s[1] = bad ? 1 : 0;
      }
    }
    if (has_w) w.load();
  } else {
    int b;
    if (!find_append_group(tok_off, first_pos, n_seq, m, grp, &b, &j)) return;  // past the last group
    seq_b = b;
    const int64_t seg0 = tok_off[b], fp = first_pos[b];
    prow = pool_off[b] + j;
    if (prow >= pool_off[b + 1]) {
      if (tid == 0) set_flag(flags, CSA2_FLAG_BAD_SEGMENT);
      return;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (u < m) {
        const int64_t pos = j * m + u;
        if (pos < fp) {  // an earlier call's token, waiting in the state
          const int64_t slot = (int64_t)b * m + pos % m;
          rw[u] = *reinterpret_cast<const uint32_t*>(st_raw + slot * kDim + c0);
          gv[u] = m > 1 ? *reinterpret_cast<const float2*>(st_gate + slot * kDim + c0) : make_float2(0.f, 0.f);
        } else {
          const int64_t tok = seg0 + (pos - fp);
          rw[u] = *reinterpret_cast<const uint32_t*>(raw + tok * kDim + c0);
          gv[u] = m > 1 ? *reinterpret_cast<const float2*>(gate + tok * kDim + c0) : make_float2(0.f, 0.f);
        }
      }
    }
    if (tail_on && tid < tail.n_query) {
      sq = tail.seq_of_q[tid];
      nvq = tail.n_vis[tid];
    }
    if (has_w) w.load();
  }
  // ---- pooling (fp32): per channel softmax of the gate logits over the group
  float pooled[2];
  if (m == 1) {
    pooled[0] = bf16lo(rw[0]);
    pooled[1] = bf16hi(rw[0]);
  } else {
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (u < m) {
        mx0 = fmaxf(mx0, gv[u].x);
        mx1 = fmaxf(mx1, gv[u].y);
      }
    }
    float d0 = 0.f, d1 = 0.f, n0 = 0.f, n1 = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (u < m) {
        const float e0 = expf(gv[u].x - mx0), e1 = expf(gv[u].y - mx1);
        d0 += e0;
        d1 += e1;
        n0 = fmaf(e0, bf16lo(rw[u]), n0);
        n1 = fmaf(e1, bf16hi(rw[u]), n1);
      }
    }
    pooled[0] = n0 / d0;
    pooled[1] = n1 / d1;
  }
  // ---- RMSNorm with norm_w
  float ss = pooled[0] * pooled[0] + pooled[1] * pooled[1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red_s[warp] = ss;
  __syncthreads();
  if (!append) {
    if (segb_s[1]) {  // the same for every thread: the CTA returns as one
      if (tid == 0) set_flag(flags, CSA2_FLAG_BAD_SEGMENT);
      return;
    }
    j = seg_s[0];
    prow = seg_s[1];
    seq_b = segb_s[0];
  }
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red_s[w];
  const float inv = 1.0f / sqrtf(tot / (float)kDim + eps);
  float ch[2] = {pooled[0] * inv * nw.x, pooled[1] * inv * nw.y};
  // ---- index key from the unrotated latent
  if (has_w) {
    *reinterpret_cast<float2*>(&c_hat_s[c0]) = make_float2(ch[0], ch[1]);
    __syncthreads();
    float cv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) cv[k] = c_hat_s[16 * lane + k];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      uint4 wau, wbu;
      w.get(u, wau, wbu);
      float acc = 0.f;
      acc = fmaf(cv[0], bf16lo(wau.x), acc); acc = fmaf(cv[1], bf16hi(wau.x), acc);
      acc = fmaf(cv[2], bf16lo(wau.y), acc); acc = fmaf(cv[3], bf16hi(wau.y), acc);
      acc = fmaf(cv[4], bf16lo(wau.z), acc); acc = fmaf(cv[5], bf16hi(wau.z), acc);
      acc = fmaf(cv[6], bf16lo(wau.w), acc); acc = fmaf(cv[7], bf16hi(wau.w), acc);
      acc = fmaf(cv[8], bf16lo(wbu.x), acc); acc = fmaf(cv[9], bf16hi(wbu.x), acc);
      acc = fmaf(cv[10], bf16lo(wbu.y), acc); acc = fmaf(cv[11], bf16hi(wbu.y), acc);
      acc = fmaf(cv[12], bf16lo(wbu.z), acc); acc = fmaf(cv[13], bf16hi(wbu.z), acc);
      acc = fmaf(cv[14], bf16lo(wbu.w), acc); acc = fmaf(cv[15], bf16hi(wbu.w), acc);
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
      if (lane == 0) k_lin_s[warp * 16 + u] = acc;
    }
    __syncthreads();
    // RMSNorm of the key; warps 0..3 own outputs [32w, 32w+32) (one fp8 block each)
    if (warp < idx_dim / 32) {
      float kss = 0.f;
      for (int o = lane; o < idx_dim; o += 32) kss += k_lin_s[o] * k_lin_s[o];
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) kss += __shfl_xor_sync(0xffffffffu, kss, sh);
      const float kinv = 1.0f / sqrtf(kss / (float)idx_dim + eps);
      const int o = warp * 32 + lane;
      const float kv = k_lin_s[o] * kinv * knw;
      if constexpr (IKF == 0) {
        const uint32_t bits = pack_bf16(kv, 0.f) & 0xFFFFu;
        reinterpret_cast<uint16_t*>(idx_keys)[prow * idx_dim + o] = (uint16_t)bits;
        k_st_s[o] = bf16lo(bits);
      } else if constexpr (IKF == 1) {
        float amax = fabsf(kv);
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
        const uint32_t eb = fp8_scale_byte(amax);
        const uint8_t code = f32_to_e4m3(ldexpf(kv, 127 - (int)eb));
        reinterpret_cast<uint8_t*>(idx_keys)[prow * idx_dim + o] = code;
        if (lane == 0) idx_key_scale[prow * (idx_dim / 32) + warp] = (uint8_t)eb;
        k_st_s[o] = e4m3_value(code) * ue8m0_value(eb);
      }
      else {
        // mxfp4: this warp's 32 outputs are one scale block; lanes 2i, 2i+1 share a byte
        float amax = fabsf(kv);
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
        const uint32_t eb = mxfp4_scale_byte(amax);
        const uint32_t code = e2m1_code(kv, ue8m0_value(eb));
        const uint32_t partner = __shfl_xor_sync(0xffffffffu, code, 1);
        if ((lane & 1) == 0) reinterpret_cast<uint8_t*>(idx_keys)[prow * (idx_dim / 2) + o / 2] = (uint8_t)(code | (partner << 4));
        if (lane == 0) idx_key_scale[prow * (idx_dim / 32) + warp] = (uint8_t)eb;
        k_st_s[o] = e2m1x2_to_float2_scaled(code).x * kE2M1Unscale * ue8m0_value(eb);
      }
    }
    if (tail_on) {
      // this entry's scores for the queries of its sequence that see it: the
      // CTA lists them (256 queries at a time), then warp w scores list
      // entries w, w + 8, ...; lane l takes channels 4l .. 4l+3 of every head,
      // with all heads' loads issued before the first is used
      const int64_t plen = pool_off[seq_b + 1] - pool_off[seq_b];
      const int64_t vis_cap = min(plen, tail.max_vis);
      for (int q0 = 0; q0 < tail.n_query; q0 += kCmpThreads) {
        const int q = q0 + tid;
        if (q0 > 0 && q < tail.n_query) {
          sq = tail.seq_of_q[q];
          nvq = tail.n_vis[q];
        }
        if (q < tail.n_query && sq == seq_b && j < min((int64_t)max(nvq, 0), vis_cap)) tq_s[atomicAdd(&tq_n, 1)] = q;
        __syncthreads();  // the list, and (first pass) the stored key's values
        const int n_list = tq_n;
        const float4 kk = *reinterpret_cast<const float4*>(&k_st_s[4 * lane]);
        for (int i = warp; i < n_list; i += kCmpThreads / 32) {
          const int qq = tq_s[i];
          const uint16_t* qrow = tail.q_idx + (int64_t)qq * tail.idx_heads * kIdxDim + 4 * lane;
          const float* wrow = tail.w_heads + (int64_t)qq * tail.idx_heads;
          float sigma = 0.f;
          for (int h0 = 0; h0 < tail.idx_heads; h0 += 8) {
            uint2 v[8];
            float wh[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const bool on = h0 + u < tail.idx_heads;
              v[u] = on ? *reinterpret_cast<const uint2*>(qrow + (int64_t)(h0 + u) * kIdxDim) : make_uint2(0u, 0u);
              wh[u] = on ? wrow[h0 + u] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (h0 + u < tail.idx_heads) {
                float d = bf16lo(v[u].x) * kk.x;
                d = fmaf(bf16hi(v[u].x), kk.y, d);
                d = fmaf(bf16lo(v[u].y), kk.z, d);
                d = fmaf(bf16hi(v[u].y), kk.w, d);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                sigma = fmaf(wh[u], fmaxf(d, 0.f), sigma);
              }
            }
          }
          if (lane == 0) tail.scores[(int64_t)qq * tail.ld + j] = sigma;
        }
        if (q0 + kCmpThreads < tail.n_query) {  // another pass: every thread has read the list
          __syncthreads();
          if (tid == 0) tq_n = 0;
          __syncthreads();
        }
      }
    }
  }
  // ---- RoPE at the group's first token position, then store
  if (rp.pairs > 0 && c0 >= kDim - 2 * rp.pairs) {
    float cs, sn;
    rope_cs(rp, (c0 - (kDim - 2 * rp.pairs)) >> 1, j * m, cs, sn);  // the group's first position
    const float x0 = ch[0], x1 = ch[1];
    ch[0] = x0 * cs - x1 * sn;
    ch[1] = x0 * sn + x1 * cs;
  }
  if constexpr (KVF == 0) {
    *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(pool_kv) + prow * kDim + c0) = pack_bf16(ch[0], ch[1]);
  } else if constexpr (KVF == 1) {
    float amax = fmaxf(fabsf(ch[0]), fabsf(ch[1]));
#pragma unroll
    for (int sh = 1; sh < 16; sh <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
    const uint32_t eb = fp8_scale_byte(amax);
    const int sh = 127 - (int)eb;
    const uint32_t word = (uint32_t)f32_to_e4m3(ldexpf(ch[0], sh)) | ((uint32_t)f32_to_e4m3(ldexpf(ch[1], sh)) << 8);
    *reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(pool_kv) + prow * kDim + c0) = (uint16_t)word;
    if ((tid & 15) == 0) pool_kv_scale[prow * (kDim / 32) + tid / 16] = (uint8_t)eb;
  } else {
    // fp4: 16 channels (8 threads) per e4m3 scale; the thread's two channels share a byte
    float amax = fmaxf(fabsf(ch[0]), fabsf(ch[1]));
#pragma unroll
    for (int sh = 1; sh < 8; sh <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
    const uint32_t sb = fp4_scale_e4m3(amax);
    const float sc = e4m3_value(sb);
    reinterpret_cast<uint8_t*>(pool_kv)[prow * (kDim / 2) + tid] =
        (uint8_t)(e2m1_code(ch[0], sc) | (e2m1_code(ch[1], sc) << 4));
    if ((tid & 7) == 0) pool_kv_scale[prow * (kDim / 16) + tid / 8] = (uint8_t)sb;
  }
}

// KVF: pool rows 0 bf16, 1 fp8, 2 fp4 (e4m3 / 16); IKF: keys 0 bf16, 1 fp8, 3 mxfp4.
// st_raw set: the append form (csa2_compress_append), tokens of a group's
// positions below first_pos[b] come from the state (slot b m + pos mod m).
// One CTA per group; WREG: the index-key weights held in registers.
template <int KVF, int IKF, bool WREG>
__global__ void __launch_bounds__(kCmpThreads) compress_kernel(const CmpArgs A, const uint16_t* __restrict__ w_idx,
                                                               const float* __restrict__ norm_w,
                                                               const float* __restrict__ k_norm_w,
                                                               const CompressTail tail) {
  // As a step's first kernel it may be launched programmatically: it reads
  // nothing before the previous kernel of the stream has finished (a plain
  // launch returns at once), which hides only the launch latency.
  pdl_wait();
  pdl_trigger();  // the step's index scan starts beside this grid
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float2 nw = *reinterpret_cast<const float2*>(norm_w + 2 * tid);
  const float knw = (w_idx != nullptr && warp < A.idx_dim / 32) ? k_norm_w[warp * 32 + lane] : 0.f;
  if constexpr (WREG) {
    CmpWRegs w;
    w.w = w_idx;
    compress_group<KVF, IKF>(A, (int64_t)blockIdx.x, w_idx != nullptr, w, nw, knw, tail);
  } else {
    CmpWGlobal w{w_idx};
    compress_group<KVF, IKF>(A, (int64_t)blockIdx.x, w_idx != nullptr, w, nw, knw, tail);
  }
}

// The append form's second launch: the new tokens of each sequence's group
// still open after the call (positions from floor((p + n) / m) m on) go to
// their state slots b m + pos mod m. One warp per new token: 1 KiB of raw
// (bf16) and 2 KiB of gate logits.
__global__ void __launch_bounds__(256) compress_state_store_kernel(
    const uint16_t* __restrict__ raw, const float* __restrict__ gate, int m, int n_seq,
    const int64_t* __restrict__ tok_off, const int64_t* __restrict__ first_pos, int64_t n_tokens,
    uint16_t* __restrict__ st_raw, float* __restrict__ st_gate) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tok = (int64_t)blockIdx.x * 8 + warp;
  if (tok >= n_tokens) return;
  const int b = find_segment_warp(tok_off, n_seq, tok);
  const int64_t p = first_pos[b], n = tok_off[b + 1] - tok_off[b];
  if (p < 0 || n < 0) return;
  const int64_t pos = p + (tok - tok_off[b]);
  if (pos < ((p + n) / m) * m) return;  // consumed by a group this call closed
  const int64_t slot = (int64_t)b * m + pos % m;
  const uint4* sr = reinterpret_cast<const uint4*>(raw + tok * kDim);
  uint4* dr = reinterpret_cast<uint4*>(st_raw + slot * kDim);
  dr[lane] = sr[lane];
  dr[lane + 32] = sr[lane + 32];
  const uint4* sg = reinterpret_cast<const uint4*>(gate + tok * kDim);
  uint4* dg = reinterpret_cast<uint4*>(st_gate + slot * kDim);
#pragma unroll
  for (int k = 0; k < 4; ++k) dg[lane + 32 * k] = sg[lane + 32 * k];
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_store_rows(cudaStream_t st, const float* rows, int64_t n_rows, int dim, const int64_t* pos,
                              const RopeParams& rp, int fmt, void* out, uint8_t* out_scale) {
  if (n_rows == 0) return cudaSuccess;
  const int rows_per_block = 8;
  const dim3 grid((unsigned)((n_rows + rows_per_block - 1) / rows_per_block));
#define CSA2_STORE(D, F) store_rows_kernel<D, F><<<grid, 256, 0, st>>>(rows, n_rows, pos, rp, out, out_scale)
  if (dim == 512) {
    switch (fmt) {
      case 0: CSA2_STORE(512, 0); break;
      case 1: CSA2_STORE(512, 1); break;
      case 2: CSA2_STORE(512, 2); break;
      case 3: CSA2_STORE(512, 3); break;
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (fmt) {
      case 0: CSA2_STORE(128, 0); break;
      case 1: CSA2_STORE(128, 1); break;
      case 2: CSA2_STORE(128, 2); break;
      case 3: CSA2_STORE(128, 3); break;
      default: return cudaErrorInvalidValue;
    }
  }
#undef CSA2_STORE
  return cudaGetLastError();
}

cudaError_t launch_compress(cudaStream_t st, int64_t n_groups, const uint16_t* raw, const float* gate, int m,
                            int n_seq, const int64_t* tok_off, const int64_t* first_pos,
                            const int64_t* pool_off, const float* norm_w, const uint16_t* w_idx,
                            const float* k_norm_w, int idx_dim, float eps, const RopeParams& rp, int kv_fmt,
                            int idx_fmt, void* pool_kv, uint8_t* pool_kv_scale, void* idx_keys,
                            uint8_t* idx_key_scale, uint32_t* flags, const AppendArgs* app, int* n_launch,
                            const CompressTail* tail, bool pdl, int num_sms) {
  if (n_groups == 0) return cudaSuccess;
  const CompressTail tl = (tail != nullptr && w_idx != nullptr) ? *tail : CompressTail{};
  const int append = app != nullptr ? 1 : 0;
  CmpArgs A{};
  A.raw = raw;
  A.gate = gate;
  A.m = m;
  A.n_seq = n_seq;
  A.tok_off = tok_off;
  A.first_pos = first_pos;
  A.pool_off = pool_off;
  A.idx_dim = idx_dim;
  A.eps = eps;
  A.rp = rp;
  A.pool_kv = pool_kv;
  A.pool_kv_scale = pool_kv_scale;
  A.idx_keys = idx_keys;
  A.idx_key_scale = idx_key_scale;
  A.flags = flags;
  A.append = append;
  A.st_raw = app != nullptr ? app->state_raw : nullptr;
  A.st_gate = app != nullptr ? app->state_gate : nullptr;
  // More than four groups an SM: the index-key weights are loaded where they
  // are used, so that two CTAs fit an SM
  const bool wreg = !(num_sms > 0 && n_groups > 4 * (int64_t)num_sms);
  cudaError_t le = cudaSuccess;
#define CSA2_COMPRESS(KF, IF)                                                                                     \
  do {                                                                                                            \
    if (wreg)                                                                                                     \
      le = launch_ex(compress_kernel<KF, IF, true>, dim3((unsigned)n_groups), dim3(kCmpThreads), 0, st, pdl, 0, A, \
                     w_idx, norm_w, k_norm_w, tl);                                                                \
    else                                                                                                          \
      le = launch_ex(compress_kernel<KF, IF, false>, dim3((unsigned)n_groups), dim3(kCmpThreads), 0, st, pdl, 0,   \
                     A, w_idx, norm_w, k_norm_w, tl);                                                             \
  } while (0)
#define CSA2_COMPRESS_K(KF)                               \
  do {                                                    \
    if (idx_fmt == 1) CSA2_COMPRESS(KF, 1);               \
    else if (idx_fmt == 3) CSA2_COMPRESS(KF, 3);          \
    else CSA2_COMPRESS(KF, 0);                            \
  } while (0)
  if (kv_fmt == 1) CSA2_COMPRESS_K(1);
  else if (kv_fmt == 2) CSA2_COMPRESS_K(2);
  else CSA2_COMPRESS_K(0);
#undef CSA2_COMPRESS_K
#undef CSA2_COMPRESS
  cudaError_t e = le != cudaSuccess ? le : cudaGetLastError();
  if (e != cudaSuccess) return e;
  *n_launch += 1;
  if (append && m > 1 && app->n_tokens > 0) {
    const dim3 g2((unsigned)((app->n_tokens + 7) / 8));
    compress_state_store_kernel<<<g2, 256, 0, st>>>(raw, gate, m, n_seq, tok_off, first_pos, app->n_tokens,
                                                    app->state_raw, app->state_gate);
    e = cudaGetLastError();
    if (e == cudaSuccess) *n_launch += 1;
  }
  return e;
}

// ---------------------------------------------------------------------------
// Staging copy of a step input that sits in page-locked host memory the device
// can address: SMs read it over the host link and write it to device memory.
// The copy engines are starved while the index scan holds the memory system,
// loads issued by SMs are not. Eight 16-byte loads in flight per thread.
constexpr int kStageThreads = 256;
constexpr int kStageUnroll = 8;

__global__ void __launch_bounds__(kStageThreads) stage_copy_kernel(const uint4* __restrict__ src,
                                                                   uint4* __restrict__ dst, int64_t n16) {
  const int64_t stride = (int64_t)gridDim.x * kStageThreads;
  int64_t i = (int64_t)blockIdx.x * kStageThreads + threadIdx.x;
  for (; i + (kStageUnroll - 1) * stride < n16; i += kStageUnroll * stride) {
    uint4 v[kStageUnroll];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

cudaError_t launch_stage_copy(cudaStream_t st, int num_sms, const void* src, void* dst, int64_t bytes,
                              int* n_launch) {
  const int64_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  // about 4 KiB per thread-round: enough loads in flight to cover the link's
  // latency, few enough CTAs to leave the index scan its SMs
  const int64_t want = (n16 + (int64_t)kStageThreads * kStageUnroll - 1) / ((int64_t)kStageThreads * kStageUnroll);
  const int64_t cap = num_sms / 4 > 0 ? num_sms / 4 : 1;
  const dim3 grid((unsigned)(want < 1 ? 1 : (want < cap ? want : cap)));
  stage_copy_kernel<<<grid, kStageThreads, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) *n_launch += 1;
  return e;
}

}  // namespace csa2
