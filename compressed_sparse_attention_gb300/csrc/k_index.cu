// Lightning-indexer scores: sigma(j) = sum_h w_h * relu(q^I_h . k^I_j)
// ("Reading Notes of DeepSeek-V4.1-Flash", section 3f, C2 step 2).
//
// The scan over the key pool is HBM-bound: one bf16 key (256 B) carries
// 8 heads x 128 x 2 = 2048 flop (8 flop/B), which fp32 FMA on the CUDA cores
// cannot sustain at full HBM rate, so the dot products go through warp-level
// mma.sync m16n8k16 (keys = 16-row A tile, the indexer query = 8-column B
// tile, fp32 accumulate). A warp streams 16-key tiles straight from global
// memory into its A fragments with 16-byte loads; because a dot product does
// not depend on the order of its terms, the k-index of the fragment is a
// fixed permutation of the channel index, applied identically to the key and
// the query fragments.
#include "launchers.cuh"

namespace csa2 {

constexpr int kIdxChunk = 256;  // keys per work item of the bf16 scan: 16 tiles, 2 per warp

// Entries [0, n) of query q that the scan covers: n_vis clamped to the pool
// and to max_vis (a larger n_vis is flagged), and, when the step scores the
// entries it compresses separately (new_first set), only the entries that
// existed before this step: those below first_pos[b] / m of a sequence that
// closes a group now.
__device__ __forceinline__ int idx_query_range(const IdxArgs& a, int q, int b, bool flag_thread, int* n_all) {
  int nv = a.n_vis[q];
  const int64_t plen = a.pool_off[b + 1] - a.pool_off[b];
  if (nv > plen || nv > a.max_vis) {
    if (flag_thread) set_flag(a.flags, CSA2_FLAG_NVIS_TOO_LARGE);
    nv = (int)min(plen, a.max_vis);
  }
  if (nv < 0) nv = 0;
  *n_all = nv;
  if (a.new_first != nullptr && a.new_tok[b + 1] > a.new_tok[b]) nv = (int)min((int64_t)nv, a.new_first[b] / a.m);
  if (a.cand != nullptr) {
    // pool form: the kept blocks hold B (kept - 1) full blocks ahead of the
    // pinned newest block, which holds the entries from B (nb - 1) on
    const int sh = a.cand_shift;
    const int nb = (nv + (1 << sh) - 1) >> sh;
    nv = nb == 0 ? 0 : ((min(nb, a.cand_ld) - 1) << sh) + (nv - ((nb - 1) << sh));
    if (flag_thread) a.n_pool[q] = nv;
  }
  return nv;
}

// key row (relative to the sequence's pool) of row position p of query q
__device__ __forceinline__ int64_t idx_row(const IdxArgs& a, int q, int64_t p) {
  if (a.cand == nullptr) return p;
  const int sh = a.cand_shift;
  return ((int64_t)a.cand[(int64_t)q * a.cand_ld + (p >> sh)] << sh) | (p & ((1 << sh) - 1));
}

// Per-query metadata a scan CTA reads at every query switch: the key row
// offset of the query's sequence, the entries it covers (n) and whether the
// sequence index is valid. Switching query every work item (64K decode: a
// CTA's items lie about five queries apart) would otherwise wait on two
// dependent loads (seq_of_q, then pool_off) before any key could be loaded;
// with the table in shared memory (filled once per CTA, every query's loads
// in flight together) the key loads of an item issue at once. Batches of up
// to kIdxMetaCap queries use it. The flags and pool counts that
// idx_query_range records are written by CTA 0 only.
constexpr int kIdxMetaCap = 256;
struct IdxMeta {
  int64_t off;  // pool_off[b]
  int32_t n;    // entries covered, 0 when the sequence index is invalid
  int32_t ok;   // sequence index valid
};
__device__ __forceinline__ void idx_fill_meta(const IdxArgs& a, IdxMeta* meta) {
  for (int q = threadIdx.x; q < a.n_query; q += blockDim.x) {
    const int b = a.seq_of_q[q];
    IdxMeta m{0, 0, 0};
    if (b >= 0 && b < a.n_seq) {
      int n_all;
      m.off = a.pool_off[b];
      m.n = idx_query_range(a, q, b, blockIdx.x == 0, &n_all);
      m.ok = 1;
    } else if (blockIdx.x == 0) {
      set_flag(a.flags, CSA2_FLAG_BAD_QUERY);
      if (a.n_pool != nullptr) a.n_pool[q] = 0;
    }
    meta[q] = m;
  }
  __syncthreads();
}

// Work items: each CTA first takes three quarters of its even share by
// striding (items c, c + G, ...; no synchronisation), then the rest is handed
// out by a 64-bit ticket counter, so that a CTA that started late (its SM
// still held by a kernel running beside the scan) just takes fewer of them.
// In the ticket phase thread 0 fetches the next ticket while the current item
// is processed; the last CTA to finish puts the counters back to zero.
__device__ __forceinline__ int64_t idx_static_items(int64_t n_items) {
  return (n_items / gridDim.x) * 3 / 4 * gridDim.x;  // the strided phase covers items [0, this)
}
// The strided phase in blocks of B consecutive items when a CTA's share
// K = n_static / gridDim.x is at least 8 (B the largest divisor of K that is
// at most 4): a CTA then switches query about once a block instead of once an
// item, and every CTA still takes exactly K items. With fewer items a CTA
// strided single items measured faster (64K decode: 25.8 against 26.2 us; at
// 1M, blocks of 3: 59.4 against 61.7 us).
__device__ __forceinline__ int idx_static_block(int64_t n_static) {
  const int64_t K = n_static / gridDim.x;
  if (K < 8) return 1;
  return K % 4 == 0 ? 4 : (K % 3 == 0 ? 3 : (K % 2 == 0 ? 2 : 1));
}

// work item -> query: items stay below 2^32 (the launcher checks), so a
// 32-bit division does (a 64-bit one costs a few hundred cycles per item)
__device__ __forceinline__ int idx_item_query(unsigned long long item, unsigned long long n_chunks) {
  return (int)((uint32_t)item / (uint32_t)n_chunks);
}

struct IdxTickets {
  unsigned long long* s;  // shared [2]
  unsigned long long* work;
  unsigned long long base;      // first ticketed item
  unsigned long long n_chunks;  // items a query (by value: the launch arguments are not addressed)
  int par = 0;
  __device__ unsigned long long draw() { return base + atomicAdd(work, 1ull); }
  // The item just run had no entries, so neither have its query's later chunks
  // (a ragged batch): the counter jumps to the next query's first item. It
  // only moves forward, so no item with entries is skipped. A test at every
  // draw was measured slower on full-length rows.
  __device__ void skip_query(unsigned long long item) {
    if (threadIdx.x == 0) {
      const int q = idx_item_query(item, n_chunks);
      atomicMax(work, (unsigned long long)(q + 1) * n_chunks - base);
    }
  }
  __device__ void start() {
    if (threadIdx.x == 0) s[0] = draw();
    __syncthreads();
  }
  __device__ unsigned long long cur() const { return s[par]; }
  __device__ void prefetch() {
    if (threadIdx.x == 0) s[par ^ 1] = draw();
  }
  __device__ void advance() {
    __syncthreads();
    par ^= 1;
  }
  __device__ void finish() {
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(work + 1, 1ull) == (unsigned long long)gridDim.x - 1ull) {
        work[0] = 0ull;
        work[1] = 0ull;
      }
    }
  }
};

// bf16 keys --------------------------------------------------------------
// Thread (g = lane/4, t = lane%4) loads, for key rows g and g+8 of a tile,
// the 16-byte chunks t, t+4, t+8, t+12 (8 channels each). In mma step
// c = 2i + h (i = chunk slot, h = half) the logical k pair (2t, 2t+1) is
// channels 8(t+4i)+4h+{0,1} and (2t+8, 2t+9) is 8(t+4i)+4h+{2,3}.
template <int NT>
__global__ void __launch_bounds__(256, 2) index_score_bf16_kernel(const IdxArgs a) {
  constexpr int HI = NT * 8;
  __shared__ unsigned long long s_tk[2];
  __shared__ IdxMeta s_meta[kIdxMetaCap];
  if (a.wait_first) pdl_wait();  // a step's first kernel, launched programmatically
  pdl_trigger();  // the step's top-k may take SMs as this grid's CTAs retire
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t n_items = a.n_chunks * (int64_t)a.n_query;
  const uint16_t* keys = reinterpret_cast<const uint16_t*>(a.keys);
  const bool use_meta = a.n_query <= kIdxMetaCap;
  if (use_meta) idx_fill_meta(a, s_meta);
  int cur_q = -1;
  uint32_t qb[NT][8][2];
  float w0[NT], w1[NT];
  int nv = 0;
  const uint16_t* kbase = nullptr;
  bool q_ok = false;
  auto run = [&](int64_t item) -> bool {  // true: the item held entries
    const int q = idx_item_query((unsigned long long)item, (unsigned long long)a.n_chunks);
    const int64_t j0 = (item - (int64_t)q * a.n_chunks) * kIdxChunk;
    if (q != cur_q) {
      cur_q = q;
      if (use_meta) {
        const IdxMeta m = s_meta[q];
        q_ok = m.ok != 0;
        nv = m.n;
        kbase = keys + m.off * kIdxDim;
      } else {
        const int b = a.seq_of_q[q];
        q_ok = (b >= 0 && b < a.n_seq);
        if (!q_ok) {
          if (threadIdx.x == 0 && j0 == 0) {
            set_flag(a.flags, CSA2_FLAG_BAD_QUERY);
            if (a.n_pool != nullptr) a.n_pool[q] = 0;
          }
        } else {
          int n_all;
          nv = idx_query_range(a, q, b, threadIdx.x == 0 && j0 == 0, &n_all);
          kbase = keys + a.pool_off[b] * kIdxDim;
        }
      }
      if (q_ok) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint16_t* qh = a.q_idx + ((int64_t)q * HI + nt * 8 + g) * kIdxDim;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(qh + 8 * (t + 4 * i));
            qb[nt][2 * i][0] = v.x; qb[nt][2 * i][1] = v.y;
            qb[nt][2 * i + 1][0] = v.z; qb[nt][2 * i + 1][1] = v.w;
          }
          w0[nt] = a.w_heads[(int64_t)q * HI + nt * 8 + 2 * t];
          w1[nt] = a.w_heads[(int64_t)q * HI + nt * 8 + 2 * t + 1];
        }
      }
    }
    if (q_ok && j0 < nv) {
      // two tiles per warp: rows j0 + 16*warp + {0..15} and j0 + 128 + 16*warp + {0..15}
      uint4 ka[2][4], kb[2][4];
      int64_t rg[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        rg[u] = j0 + 128 * u + 16 * warp + g;
        const int64_t ra = idx_row(a, q, min(rg[u], (int64_t)nv - 1));
        const int64_t rb = idx_row(a, q, min(rg[u] + 8, (int64_t)nv - 1));
        const uint16_t* pa = kbase + ra * kIdxDim;
        const uint16_t* pb = kbase + rb * kIdxDim;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ka[u][i] = ldg_stream16(pa + 8 * (t + 4 * i));
          kb[u][i] = ldg_stream16(pb + 8 * (t + 4 * i));
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float sg = 0.f, sg8 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            mma_16816_bf16(acc, ka[u][i].x, kb[u][i].x, ka[u][i].y, kb[u][i].y, qb[nt][2 * i][0], qb[nt][2 * i][1]);
            mma_16816_bf16(acc, ka[u][i].z, kb[u][i].z, ka[u][i].w, kb[u][i].w, qb[nt][2 * i + 1][0],
                           qb[nt][2 * i + 1][1]);
          }
          sg = fmaf(w0[nt], fmaxf(acc[0], 0.f), sg);
          sg = fmaf(w1[nt], fmaxf(acc[1], 0.f), sg);
          sg8 = fmaf(w0[nt], fmaxf(acc[2], 0.f), sg8);
          sg8 = fmaf(w1[nt], fmaxf(acc[3], 0.f), sg8);
        }
        sg += __shfl_xor_sync(0xffffffffu, sg, 1);
        sg += __shfl_xor_sync(0xffffffffu, sg, 2);
        sg8 += __shfl_xor_sync(0xffffffffu, sg8, 1);
        sg8 += __shfl_xor_sync(0xffffffffu, sg8, 2);
        float* srow = a.scores + (int64_t)q * a.ld;
        if (t == 0 && rg[u] < nv) srow[rg[u]] = sg;
        if (t == 1 && rg[u] + 8 < nv) srow[rg[u] + 8] = sg8;
      }
    }
    return q_ok && j0 < nv;
  };
  const int64_t n_static = idx_static_items(n_items);
  {
    const int B = idx_static_block(n_static);
    for (int64_t blk = blockIdx.x; blk * B < n_static; blk += gridDim.x)
      for (int k = 0; k < B; ++k) run(blk * B + k);
  }
  IdxTickets tk{s_tk, a.work, (unsigned long long)n_static, (unsigned long long)a.n_chunks};
  tk.start();
  for (;;) {
    const unsigned long long item = tk.cur();
    if (item >= (unsigned long long)n_items) break;
    tk.prefetch();
    if (!run((int64_t)item)) tk.skip_query(item);
    tk.advance();
  }
  tk.finish();
  pdl_wait();  // launched after compress: this grid ends only once compress has
}

// fp8 / mxfp4 keys ---------------------------------------------------------
// A key row is 128 codes (e4m3: 128 B; E2M1: two to a byte, 64 B) plus 4
// ue8m0 scales, one per 32 channels. Thread (g, t) reads the codes of
// channels 32b + 8t .. +7 of rows g and g+8 for each block b, so an mma step
// never mixes two scale blocks; each block's partial dot product is scaled by
// its power of two in fp32.
//
// Both code types decode exactly into f16 with one hardware conversion per
// pair of codes (e4m3x2 -> f16x2, e2m1x2 -> f16x2), so these products run as
// f16 x f16 -> f32 mma. The
// indexer query is converted to f16 once per query, head h multiplied by a
// power of two 2^s_h that puts its largest element in [2^14, 2^15): every
// bf16 element at least 2^-24 of that largest one is then exact in f16, and
// a smaller one moves by at most 2^-25 of it. The weight w_h takes the
// inverse power, which the ReLU commutes with. k-slot order (both code
// types): mma step (b, 0) holds channel pairs (8t, 8t+1) and (8t+2, 8t+3) of
// block b, step (b, 1) the pairs (8t+4, 8t+5) and (8t+6, 8t+7).
template <int NT, int KF>
__device__ __forceinline__ void idxq_load_query(const uint16_t* __restrict__ q_idx, const float* __restrict__ w_heads,
                                                int q, int g, int t, uint32_t (&qb)[NT][8][2], float (&w0)[NT],
                                                float (&w1)[NT]) {
  constexpr int HI = NT * 8;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint16_t* qh = q_idx + ((int64_t)q * HI + nt * 8 + g) * kIdxDim;
    // pass 1: the head's largest magnitude (bf16 -> float is exact)
    float amax = 0.f;
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
      const uint4 v = *reinterpret_cast<const uint4*>(qh + 32 * bb + 8 * t);
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(v.x << 16)), fabsf(__uint_as_float(v.x & 0xFFFF0000u))));
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(v.y << 16)), fabsf(__uint_as_float(v.y & 0xFFFF0000u))));
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(v.z << 16)), fabsf(__uint_as_float(v.z & 0xFFFF0000u))));
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(v.w << 16)), fabsf(__uint_as_float(v.w & 0xFFFF0000u))));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int ex = 0;
    if (amax > 0.f) frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
    const int sh = max(-100, min(100, 15 - ex));
    const float up = __uint_as_float((uint32_t)(sh + 127) << 23);
    // pass 2: scaled f16 pairs in k-slot order (the row is in L1 from pass 1)
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
      const uint4 v = *reinterpret_cast<const uint4*>(qh + 32 * bb + 8 * t);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      float y[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        y[2 * k] = __uint_as_float(wv[k] << 16) * up;
        y[2 * k + 1] = __uint_as_float(wv[k] & 0xFFFF0000u) * up;
      }
      qb[nt][2 * bb][0] = h2_bits(y[0], y[1]);
      qb[nt][2 * bb][1] = h2_bits(y[2], y[3]);
      qb[nt][2 * bb + 1][0] = h2_bits(y[4], y[5]);
      qb[nt][2 * bb + 1][1] = h2_bits(y[6], y[7]);
    }
    // the C fragment's columns are heads 2t and 2t+1, whose powers lanes 8t and 8t+4 hold
    const int e = -sh;
    const int e0 = __shfl_sync(0xffffffffu, e, 8 * t), e1 = __shfl_sync(0xffffffffu, e, 8 * t + 4);
    w0[nt] = ldexpf(w_heads[(int64_t)q * HI + nt * 8 + 2 * t], e0);
    w1[nt] = ldexpf(w_heads[(int64_t)q * HI + nt * 8 + 2 * t + 1], e1);
  }
}

// U = tiles of 16 keys per warp per work item (chunk = 128 U keys): all of a
// warp's loads for an item are issued before any is used, so U sets the bytes
// in flight (16 warps an SM x U x 16 rows x row bytes); mxfp4 rows are half
// the size of fp8 rows and take twice the tiles.
template <int NT, int KF, int U>
__global__ void __launch_bounds__(256, 2) index_score_fp8_kernel(const IdxArgs a) {
  constexpr int KB = KF == 3 ? kIdxDim / 2 : kIdxDim;  // code bytes a key
  constexpr int CH = 128 * U;                         // keys a work item
  __shared__ unsigned long long s_tk[2];
  __shared__ IdxMeta s_meta[kIdxMetaCap];
  if (a.wait_first) pdl_wait();  // a step's first kernel, launched programmatically
  pdl_trigger();  // the step's top-k may take SMs as this grid's CTAs retire
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t n_items = a.n_chunks * (int64_t)a.n_query;
  const uint8_t* keys = reinterpret_cast<const uint8_t*>(a.keys);
  const bool use_meta = a.n_query <= kIdxMetaCap;
  if (use_meta) idx_fill_meta(a, s_meta);
  int cur_q = -1;
  uint32_t qb[NT][8][2];
  float w0[NT], w1[NT];
  int nv = 0;
  const uint8_t* kbase = nullptr;
  const uint8_t* sbase = nullptr;
  bool q_ok = false;
  auto run = [&](int64_t item) -> bool {  // true: the item held entries
    const int q = idx_item_query((unsigned long long)item, (unsigned long long)a.n_chunks);
    const int64_t j0 = (item - (int64_t)q * a.n_chunks) * CH;
    if (q != cur_q) {
      cur_q = q;
      int64_t off = 0;
      if (use_meta) {
        const IdxMeta m = s_meta[q];
        q_ok = m.ok != 0;
        nv = m.n;
        off = m.off;
      } else {
        const int b = a.seq_of_q[q];
        q_ok = (b >= 0 && b < a.n_seq);
        if (!q_ok) {
          if (threadIdx.x == 0 && j0 == 0) {
            set_flag(a.flags, CSA2_FLAG_BAD_QUERY);
            if (a.n_pool != nullptr) a.n_pool[q] = 0;
          }
        } else {
          int n_all;
          nv = idx_query_range(a, q, b, threadIdx.x == 0 && j0 == 0, &n_all);
          off = a.pool_off[b];
        }
      }
      if (q_ok) {
        kbase = keys + off * KB;
        sbase = a.key_scale + off * (kIdxDim / 32);
        idxq_load_query<NT, KF>(a.q_idx, a.w_heads, q, g, t, qb, w0, w1);
      }
    }
    if (q_ok && j0 < nv) {
      // KF 3 keeps 4 code bytes per (tile, block, row) in .x; the .y words are unused
      uint2 ca[U][4], cb[U][4];
      uint32_t sa[U], sb[U];
      int64_t rg[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        rg[u] = j0 + 128 * u + 16 * warp + g;
        const int64_t ra = idx_row(a, q, min(rg[u], (int64_t)nv - 1));
        const int64_t rb = idx_row(a, q, min(rg[u] + 8, (int64_t)nv - 1));
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          if constexpr (KF == 3) {  // 8 codes in 4 bytes
            ca[u][bb] = make_uint2(ldg_stream4(kbase + ra * KB + 16 * bb + 4 * t), 0u);
            cb[u][bb] = make_uint2(ldg_stream4(kbase + rb * KB + 16 * bb + 4 * t), 0u);
          } else {
            ca[u][bb] = ldg_stream8(kbase + ra * KB + 32 * bb + 8 * t);
            cb[u][bb] = ldg_stream8(kbase + rb * KB + 32 * bb + 8 * t);
          }
        }
        sa[u] = *reinterpret_cast<const uint32_t*>(sbase + ra * 4);
        sb[u] = *reinterpret_cast<const uint32_t*>(sbase + rb * 4);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float tot[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) tot[nt][0] = tot[nt][1] = tot[nt][2] = tot[nt][3] = 0.f;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          // this block's 8 codes of rows g (a) and g+8 (b) as f16 pairs in k-slot order
          uint32_t a[4], b[4];
          if constexpr (KF == 3) {
            e2m1x8_to_f16x2x4_cvt(ca[u][bb].x, a);
            e2m1x8_to_f16x2x4_cvt(cb[u][bb].x, b);
          } else {
            a[0] = e4m3x2_to_f16x2(ca[u][bb].x); a[1] = e4m3x2_to_f16x2(ca[u][bb].x >> 16);
            a[2] = e4m3x2_to_f16x2(ca[u][bb].y); a[3] = e4m3x2_to_f16x2(ca[u][bb].y >> 16);
            b[0] = e4m3x2_to_f16x2(cb[u][bb].x); b[1] = e4m3x2_to_f16x2(cb[u][bb].x >> 16);
            b[2] = e4m3x2_to_f16x2(cb[u][bb].y); b[3] = e4m3x2_to_f16x2(cb[u][bb].y >> 16);
          }
          const float scg = ue8m0_value((sa[u] >> (8 * bb)) & 0xFFu);
          const float scg8 = ue8m0_value((sb[u] >> (8 * bb)) & 0xFFu);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816_f16(acc, a[0], b[0], a[1], b[1], qb[nt][2 * bb][0], qb[nt][2 * bb][1]);
            mma_16816_f16(acc, a[2], b[2], a[3], b[3], qb[nt][2 * bb + 1][0], qb[nt][2 * bb + 1][1]);
            tot[nt][0] = fmaf(scg, acc[0], tot[nt][0]);
            tot[nt][1] = fmaf(scg, acc[1], tot[nt][1]);
            tot[nt][2] = fmaf(scg8, acc[2], tot[nt][2]);
            tot[nt][3] = fmaf(scg8, acc[3], tot[nt][3]);
          }
        }
        float sg = 0.f, sg8 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          sg = fmaf(w0[nt], fmaxf(tot[nt][0], 0.f), sg);
          sg = fmaf(w1[nt], fmaxf(tot[nt][1], 0.f), sg);
          sg8 = fmaf(w0[nt], fmaxf(tot[nt][2], 0.f), sg8);
          sg8 = fmaf(w1[nt], fmaxf(tot[nt][3], 0.f), sg8);
        }
        sg += __shfl_xor_sync(0xffffffffu, sg, 1);
        sg += __shfl_xor_sync(0xffffffffu, sg, 2);
        sg8 += __shfl_xor_sync(0xffffffffu, sg8, 1);
        sg8 += __shfl_xor_sync(0xffffffffu, sg8, 2);
        float* srow = a.scores + (int64_t)q * a.ld;
        if (t == 0 && rg[u] < nv) srow[rg[u]] = sg;
        if (t == 1 && rg[u] + 8 < nv) srow[rg[u] + 8] = sg8;
      }
    }
    return q_ok && j0 < nv;
  };
  const int64_t n_static = idx_static_items(n_items);
  {
    const int B = idx_static_block(n_static);
    for (int64_t blk = blockIdx.x; blk * B < n_static; blk += gridDim.x)
      for (int k = 0; k < B; ++k) run(blk * B + k);
  }
  IdxTickets tk{s_tk, a.work, (unsigned long long)n_static, (unsigned long long)a.n_chunks};
  tk.start();
  for (;;) {
    const unsigned long long item = tk.cur();
    if (item >= (unsigned long long)n_items) break;
    tk.prefetch();
    if (!run((int64_t)item)) tk.skip_query(item);
    tk.advance();
  }
  tk.finish();
  pdl_wait();  // launched after compress: this grid ends only once compress has
}

cudaError_t launch_index_score(cudaStream_t st, int num_sms, int idx_heads, int idx_fmt, IdxArgs a, bool pdl) {
  if (a.n_query == 0 || a.max_vis == 0) return cudaSuccess;
  const int64_t cap = (int64_t)num_sms * 2;
  // chunk of one work item: 256 keys (bf16; fp8 and mxfp4 with 32 heads), 512
  // (fp8 with 8 heads, mxfp4 with 8 or 16 heads)
  const int u_q = ((idx_fmt == 3 && idx_heads <= 16) || (idx_fmt == 1 && idx_heads == 8)) ? 4 : 2;
  const int64_t chunk = idx_fmt == 0 ? kIdxChunk : 128 * u_q;
  const int64_t rows_max = a.cand != nullptr ? min(a.max_vis, (int64_t)a.cand_ld << a.cand_shift) : a.max_vis;
  a.n_chunks = (rows_max + chunk - 1) / chunk;
  const int64_t items = a.n_chunks * a.n_query;
  if (items >= (int64_t)1 << 32) return cudaErrorInvalidValue;  // item indices are split in 32 bits
  const dim3 grid((unsigned)(items < cap ? items : cap));
  cudaError_t le = cudaSuccess;
#define CSA2_IDX(NT, UQ, U8)                                                                          \
  do {                                                                                                \
    if (idx_fmt == 1) le = launch_ex(index_score_fp8_kernel<NT, 1, U8>, grid, dim3(256), 0, st, pdl, 0, a); \
    else if (idx_fmt == 3)                                                                            \
      le = launch_ex(index_score_fp8_kernel<NT, 3, UQ>, grid, dim3(256), 0, st, pdl, 0, a);           \
    else le = launch_ex(index_score_bf16_kernel<NT>, grid, dim3(256), 0, st, pdl, 0, a);              \
  } while (0)
  switch (idx_heads) {
    case 8: CSA2_IDX(1, 4, 4); break;
    case 16: CSA2_IDX(2, 4, 2); break;
    case 32: CSA2_IDX(4, 2, 2); break;
    default: return cudaErrorInvalidValue;
  }
#undef CSA2_IDX
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace csa2
