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

constexpr int kIdxChunk = 256;  // keys per work item: 16 tiles, 2 per warp

// bf16 keys --------------------------------------------------------------
// Thread (g = lane/4, t = lane%4) loads, for key rows g and g+8 of a tile,
// the 16-byte chunks t, t+4, t+8, t+12 (8 channels each). In mma step
// c = 2i + h (i = chunk slot, h = half) the logical k pair (2t, 2t+1) is
// channels 8(t+4i)+4h+{0,1} and (2t+8, 2t+9) is 8(t+4i)+4h+{2,3}.
template <int NT>
__global__ void __launch_bounds__(256, 2) index_score_bf16_kernel(
    int n_query, int n_seq, int64_t n_chunks, int64_t max_vis, const uint16_t* __restrict__ q_idx,
    const float* __restrict__ w_heads, const uint16_t* __restrict__ keys,
    const int64_t* __restrict__ pool_off, const int32_t* __restrict__ seq_of_q,
    const int32_t* __restrict__ n_vis, float* __restrict__ scores, int64_t ld, uint32_t* flags) {
  constexpr int HI = NT * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t n_items = n_chunks * (int64_t)n_query;
  int cur_q = -1;
  uint32_t qb[NT][8][2];
  float w0[NT], w1[NT];
  int nv = 0;
  const uint16_t* kbase = nullptr;
  bool q_ok = false;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int q = (int)(item / n_chunks);
    const int64_t j0 = (item % n_chunks) * kIdxChunk;
    if (q != cur_q) {
      cur_q = q;
      const int b = seq_of_q[q];
      nv = n_vis[q];
      q_ok = (b >= 0 && b < n_seq);
      if (!q_ok) {
        if (threadIdx.x == 0 && j0 == 0) set_flag(flags, CSA2_FLAG_BAD_QUERY);
      } else {
        const int64_t plen = pool_off[b + 1] - pool_off[b];
        if (nv > plen || nv > max_vis) {
          if (threadIdx.x == 0 && j0 == 0) set_flag(flags, CSA2_FLAG_NVIS_TOO_LARGE);
          nv = (int)min(plen, max_vis);
        }
        kbase = keys + pool_off[b] * kIdxDim;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint16_t* qh = q_idx + ((int64_t)q * HI + nt * 8 + g) * kIdxDim;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(qh + 8 * (t + 4 * i));
            qb[nt][2 * i][0] = v.x; qb[nt][2 * i][1] = v.y;
            qb[nt][2 * i + 1][0] = v.z; qb[nt][2 * i + 1][1] = v.w;
          }
          w0[nt] = w_heads[(int64_t)q * HI + nt * 8 + 2 * t];
          w1[nt] = w_heads[(int64_t)q * HI + nt * 8 + 2 * t + 1];
        }
      }
    }
    if (!q_ok || j0 >= nv) continue;
    // two tiles per warp: rows j0 + 16*warp + {0..15} and j0 + 128 + 16*warp + {0..15}
    uint4 ka[2][4], kb[2][4];
    int64_t rg[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      rg[u] = j0 + 128 * u + 16 * warp + g;
      const int64_t ra = min(rg[u], (int64_t)nv - 1), rb = min(rg[u] + 8, (int64_t)nv - 1);
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
      float* srow = scores + (int64_t)q * ld;
      if (t == 0 && rg[u] < nv) srow[rg[u]] = sg;
      if (t == 1 && rg[u] + 8 < nv) srow[rg[u] + 8] = sg8;
    }
  }
}

// fp8 keys ---------------------------------------------------------------
// A key row is 128 e4m3 codes plus 4 ue8m0 scales (one per 32 channels).
// Thread (g, t) reads 8 codes at channels 32b + 8t .. +7 of rows g and g+8
// for each block b; mma step (b, s) covers channels 32b + 8t + 4s + {0..3},
// so one step never mixes two scale blocks. Codes convert exactly to bf16;
// each block's partial dot product is scaled by its power of two in fp32.
// KF 1: e4m3 codes (128 B a key); KF 3: E2M1 codes two to a byte (64 B a key);
// both with a ue8m0 scale per 32 channels
template <int NT, int KF>
__global__ void __launch_bounds__(256, 2) index_score_fp8_kernel(
    int n_query, int n_seq, int64_t n_chunks, int64_t max_vis, const uint16_t* __restrict__ q_idx,
    const float* __restrict__ w_heads, const uint8_t* __restrict__ keys, const uint8_t* __restrict__ key_scale,
    const int64_t* __restrict__ pool_off, const int32_t* __restrict__ seq_of_q,
    const int32_t* __restrict__ n_vis, float* __restrict__ scores, int64_t ld, uint32_t* flags) {
  constexpr int HI = NT * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t n_items = n_chunks * (int64_t)n_query;
  int cur_q = -1;
  uint32_t qb[NT][8][2];
  float w0[NT], w1[NT];
  int nv = 0;
  const uint8_t* kbase = nullptr;
  const uint8_t* sbase = nullptr;
  bool q_ok = false;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int q = (int)(item / n_chunks);
    const int64_t j0 = (item % n_chunks) * kIdxChunk;
    if (q != cur_q) {
      cur_q = q;
      const int b = seq_of_q[q];
      nv = n_vis[q];
      q_ok = (b >= 0 && b < n_seq);
      if (!q_ok) {
        if (threadIdx.x == 0 && j0 == 0) set_flag(flags, CSA2_FLAG_BAD_QUERY);
      } else {
        const int64_t plen = pool_off[b + 1] - pool_off[b];
        if (nv > plen || nv > max_vis) {
          if (threadIdx.x == 0 && j0 == 0) set_flag(flags, CSA2_FLAG_NVIS_TOO_LARGE);
          nv = (int)min(plen, max_vis);
        }
        kbase = keys + pool_off[b] * (KF == 3 ? kIdxDim / 2 : kIdxDim);
        sbase = key_scale + pool_off[b] * (kIdxDim / 32);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint16_t* qh = q_idx + ((int64_t)q * HI + nt * 8 + g) * kIdxDim;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const uint4 v = *reinterpret_cast<const uint4*>(qh + 32 * bb + 8 * t);
            qb[nt][2 * bb][0] = v.x; qb[nt][2 * bb][1] = v.y;
            qb[nt][2 * bb + 1][0] = v.z; qb[nt][2 * bb + 1][1] = v.w;
          }
          w0[nt] = w_heads[(int64_t)q * HI + nt * 8 + 2 * t];
          w1[nt] = w_heads[(int64_t)q * HI + nt * 8 + 2 * t + 1];
        }
      }
    }
    if (!q_ok || j0 >= nv) continue;
    uint2 ca[2][4], cb[2][4];
    uint32_t sa[2], sb[2];
    int64_t rg[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      rg[u] = j0 + 128 * u + 16 * warp + g;
      const int64_t ra = min(rg[u], (int64_t)nv - 1), rb = min(rg[u] + 8, (int64_t)nv - 1);
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        if constexpr (KF == 3) {  // 8 codes in 4 bytes
          ca[u][bb] = make_uint2(*reinterpret_cast<const uint32_t*>(kbase + ra * (kIdxDim / 2) + 16 * bb + 4 * t), 0u);
          cb[u][bb] = make_uint2(*reinterpret_cast<const uint32_t*>(kbase + rb * (kIdxDim / 2) + 16 * bb + 4 * t), 0u);
        } else {
          ca[u][bb] = ldg_stream8(kbase + ra * kIdxDim + 32 * bb + 8 * t);
          cb[u][bb] = ldg_stream8(kbase + rb * kIdxDim + 32 * bb + 8 * t);
        }
      }
      sa[u] = *reinterpret_cast<const uint32_t*>(sbase + ra * 4);
      sb[u] = *reinterpret_cast<const uint32_t*>(sbase + rb * 4);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float tot[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) tot[nt][0] = tot[nt][1] = tot[nt][2] = tot[nt][3] = 0.f;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        // exact e4m3 -> bf16 (or E2M1 -> 2^-14 times its value, in bf16) of
        // this block's 8 codes per row
        uint32_t a[4], b[4];
        if constexpr (KF == 3) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 fa = e2m1x2_to_float2_scaled((ca[u][bb].x >> (8 * k)) & 0xFFu);
            const float2 fb = e2m1x2_to_float2_scaled((cb[u][bb].x >> (8 * k)) & 0xFFu);
            a[k] = pack_bf16(fa.x, fa.y);
            b[k] = pack_bf16(fb.x, fb.y);
          }
        } else {
          const float2 f0 = e4m3x2_to_float2((uint16_t)(ca[u][bb].x & 0xFFFF));
          const float2 f1 = e4m3x2_to_float2((uint16_t)(ca[u][bb].x >> 16));
          const float2 f2 = e4m3x2_to_float2((uint16_t)(ca[u][bb].y & 0xFFFF));
          const float2 f3 = e4m3x2_to_float2((uint16_t)(ca[u][bb].y >> 16));
          a[0] = pack_bf16(f0.x, f0.y); a[1] = pack_bf16(f1.x, f1.y);
          a[2] = pack_bf16(f2.x, f2.y); a[3] = pack_bf16(f3.x, f3.y);
          const float2 h0 = e4m3x2_to_float2((uint16_t)(cb[u][bb].x & 0xFFFF));
          const float2 h1 = e4m3x2_to_float2((uint16_t)(cb[u][bb].x >> 16));
          const float2 h2 = e4m3x2_to_float2((uint16_t)(cb[u][bb].y & 0xFFFF));
          const float2 h3 = e4m3x2_to_float2((uint16_t)(cb[u][bb].y >> 16));
          b[0] = pack_bf16(h0.x, h0.y); b[1] = pack_bf16(h1.x, h1.y);
          b[2] = pack_bf16(h2.x, h2.y); b[3] = pack_bf16(h3.x, h3.y);
        }
        const float unscale = KF == 3 ? kE2M1Unscale : 1.0f;
        const float scg = ue8m0_value((sa[u] >> (8 * bb)) & 0xFFu) * unscale;
        const float scg8 = ue8m0_value((sb[u] >> (8 * bb)) & 0xFFu) * unscale;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          mma_16816_bf16(acc, a[0], b[0], a[1], b[1], qb[nt][2 * bb][0], qb[nt][2 * bb][1]);
          mma_16816_bf16(acc, a[2], b[2], a[3], b[3], qb[nt][2 * bb + 1][0], qb[nt][2 * bb + 1][1]);
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
      float* srow = scores + (int64_t)q * ld;
      if (t == 0 && rg[u] < nv) srow[rg[u]] = sg;
      if (t == 1 && rg[u] + 8 < nv) srow[rg[u] + 8] = sg8;
    }
  }
}

cudaError_t launch_index_score(cudaStream_t st, int num_sms, int idx_heads, int idx_fmt, int n_query, int n_seq,
                               int64_t max_vis, const uint16_t* q_idx, const float* w_heads, const void* keys,
                               const uint8_t* key_scale, const int64_t* pool_off, const int32_t* seq_of_q,
                               const int32_t* n_vis, float* scores, int64_t ld, uint32_t* flags) {
  if (n_query == 0 || max_vis == 0) return cudaSuccess;
  const int64_t n_chunks = (max_vis + kIdxChunk - 1) / kIdxChunk;
  const int64_t items = n_chunks * n_query;
  const int64_t cap = (int64_t)num_sms * 2;
  const dim3 grid((unsigned)(items < cap ? items : cap));
#define CSA2_IDX(NT)                                                                                   \
  do {                                                                                                 \
    if (idx_fmt == 1)                                                                                  \
      index_score_fp8_kernel<NT, 1><<<grid, 256, 0, st>>>(n_query, n_seq, n_chunks, max_vis, q_idx, w_heads, \
                                                       (const uint8_t*)keys, key_scale, pool_off,      \
                                                       seq_of_q, n_vis, scores, ld, flags);            \
    else if (idx_fmt == 3)                                                                             \
      index_score_fp8_kernel<NT, 3><<<grid, 256, 0, st>>>(n_query, n_seq, n_chunks, max_vis, q_idx, w_heads, \
                                                       (const uint8_t*)keys, key_scale, pool_off,      \
                                                       seq_of_q, n_vis, scores, ld, flags);            \
    else                                                                                               \
      index_score_bf16_kernel<NT><<<grid, 256, 0, st>>>(n_query, n_seq, n_chunks, max_vis, q_idx, w_heads, \
                                                        (const uint16_t*)keys, pool_off, seq_of_q,     \
                                                        n_vis, scores, ld, flags);                     \
  } while (0)
  switch (idx_heads) {
    case 8: CSA2_IDX(1); break;
    case 16: CSA2_IDX(2); break;
    case 32: CSA2_IDX(4); break;
    default: return cudaErrorInvalidValue;
  }
#undef CSA2_IDX
  return cudaGetLastError();
}

}  // namespace csa2
