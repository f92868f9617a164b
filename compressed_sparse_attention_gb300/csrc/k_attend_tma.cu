// Two-source sparse attention for bf16 rows with the rows gathered by the
// tensor memory accelerator ("Reading Notes of DeepSeek-V4.1-Flash", section
// 3a and section 3f, C2 step 3; the products, the softmax and the epilogue
// are those of attend_tile.cuh, shared with the thread-gathered kernel).
//
// A CTA holds 8 math warps and one producer warp. The producer computes each
// tile's 128 row sources (lane l: rows 4l .. 4l+3) and gathers the rows with
// `cp.async.bulk.tensor.2d ... tile::gather4`: one instruction brings 4 rows
// of one 64-channel block (128 B each) into the 128-byte-swizzled operand
// layout, a row of -1 reading zeros. A tile lands as four pairs of channel
// blocks, each pair on its own mbarrier (full[g], 32 KiB of transaction
// bytes). Its QK^T steps are issued as soon as the pair lands.
// The PV product of tile i runs as four blocks of 128 output dims. Block g
// reads only channel pair g, and its tcgen05.commit arrives on empty[g], so
// the producer refills pair g with tile i+1's rows while blocks g+1..3 still
// run. The gather of the next tile thereby overlaps the PV product of this
// one and the QK^T product of the next, and no math thread takes part in it.
// The producer also publishes each tile's row masks (one bit a row) before it
// arrives on the tile's full barriers; the math threads read them after
// waiting on full[3].
// Every wait is bounded: on a timeout the waiter records
// CSA2_FLAG_WAIT_TIMEOUT, the CTA stops issuing work and lets what is in
// flight land before it frees tensor memory.
#include "attend_tile.cuh"

#include <cuda.h>  // CUtensorMap and its encoding enums; the encoder is resolved at run time
#include <cstring>
#include <mutex>

namespace csa2 {

constexpr int kTmaThreads = kAttThreads + 32;           // 8 math warps + 1 producer warp
constexpr uint32_t kPairBytes = 2u * kTileRows * 128u;  // two 64-channel blocks of a tile: 32 KiB
// barriers and row masks in the SM_ROWS region (this kernel keeps row sources
// in the producer's registers)
constexpr uint32_t TB_S = SM_ROWS;            // S^T ready, or all tensor-core work done
constexpr uint32_t TB_FULL = SM_ROWS + 8;     // [4] channel pair g of the tile landed
constexpr uint32_t TB_EMPTY = SM_ROWS + 40;   // [4] PV block g done: pair g may be refilled
constexpr uint32_t TB_MASK = SM_ROWS + 128;   // uint32 [2][4]: row r valid = bit (r >> 2) of word r & 3

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// 4 rows (r0..r3, -1: zeros) x 64 channels from `col` of a [rows, 512] bf16
// tensor into 512 B of 128-byte-swizzled shared memory at dst
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar, int col, int r0,
                                            int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

__global__ void __launch_bounds__(kTmaThreads, 1)
    attend_tma_kernel(const AttendParams p, const __grid_constant__ CUtensorMap win_map,
                      const __grid_constant__ CUtensorMap pool_map) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_s - raw_s);
  float* m_run = reinterpret_cast<float*>(sm + SM_MRUN);
  float* l_run = reinterpret_cast<float*>(sm + SM_LRUN);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + SM_MISC);  // [2] tmem slot, [3] rescale
  uint32_t* mask = reinterpret_cast<uint32_t*>(sm + TB_MASK);
  const uint32_t s_bar = base_s + TB_S;
  const uint32_t tslot = base_s + SM_MISC + 8;

  if (p.pdl) pdl_trigger();  // the merge may take the room this grid leaves
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp == kAttWarps;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;  // a math thread's tile row / output dim in a 128 block
  // CTAs are numbered split-major (all queries' first CTAs first, which hold
  // the window tile and start before the selection exists). Split 0 takes
  // the launch's first lead_tiles tiles, the others tiles_per_split each.
  const int qi = blockIdx.x % p.n_query, split = blockIdx.x / p.n_query;
  const int lead = p.lead_tiles;
  const int tile_begin = split == 0 ? p.tile_base : p.tile_base + lead + (split - 1) * p.tiles_per_split;
  const int tile_cap0 = split == 0 ? tile_begin + lead : tile_begin + p.tiles_per_split;
  const int tile_cap = min(tile_cap0, p.tile_base + p.tile_count);
  const int64_t t = p.q_pos[qi];
  const int b = p.seq_of_q[qi];
  // Q is copied asynchronously by the math warps into its swizzled K-major slots
  if (!producer && tile_begin < tile_cap) {
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
  cp_async_commit();
  const bool q_ok = (b >= 0 && b < p.n_seq && t >= 0);
  const int tile_end = q_ok ? tile_cap : tile_begin;
  if (!q_ok && tid == 0 && split == 0) set_flag(p.flags, CSA2_FLAG_BAD_QUERY);
  const int bs = q_ok ? b : 0;  // offsets of a valid sequence (unused when !q_ok)
  const int64_t win_b0 = p.win_off != nullptr ? p.win_off[bs] : 0;
  const int64_t win_b1 = p.win_off != nullptr ? p.win_off[bs + 1] : 0;
  // no selection (window-only call): the pool arguments may be NULL
  const int64_t pool_b0 = p.pool_off != nullptr ? p.pool_off[bs] : 0;
  const int64_t pool_b1 = p.pool_off != nullptr ? p.pool_off[bs + 1] : 0;
  const int64_t lo_raw = (q_ok && p.win_lo) ? p.win_lo[bs] : 0;

  if (warp == 0) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(s_bar, 1);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      mbar_init(base_s + TB_FULL + 8 * g, 1);
      mbar_init(base_s + TB_EMPTY + 8 * g, 1);
    }
    fence_mbar_init();
    misc[3] = 0;
  }
  if (tid < kHeads) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.f;
  }
  float2* rope_tab = reinterpret_cast<float2*>(sm + SM_ROPE);
  const float sink_l2 = (p.direct == 1 && tid < kHeads) ? p.sink[tid] * 1.4426950408889634f : 0.f;  // used at the end
  if (tid < p.rp.pairs) {
    float c = 1.f, sn = 0.f;
    if (q_ok) rope_cs(p.rp, tid, t, c, sn);
    rope_tab[tid] = make_float2(c, sn);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = misc[2];
  const uint32_t tmem_s = taddr;       // columns [0, 64)
  const uint32_t tmem_o = taddr + 64;  // columns [64, 320)
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const int64_t win_cap = q_ok ? (win_b1 - win_b0) : 0;
  const int64_t lo_b = max((int64_t)0, lo_raw);
  const int64_t lo_eff = max(lo_b, t - (int64_t)p.window + 1);
  const int64_t plen = q_ok ? (pool_b1 - pool_b0) : 0;

  if (producer) {
    // ---------------- producer warp: row sources and TMA gathers
    const int32_t* sel = p.topk_idx != nullptr ? p.topk_idx + (int64_t)qi * p.topk : nullptr;
    int32_t jn[4] = {-1, -1, -1, -1};
    bool sel_waited = false;
    // this lane's 4 selection entries of selected tile `tile`; launched
    // programmatically after the step's top-k, the first read waits for it
    // (the window tile needs no selection and is gathered before)
    auto load_sel = [&](int tile) {
      if (!sel_waited) {
        pdl_wait();
        sel_waited = true;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = (tile - 1) * kTileRows + 4 * lane + j;
        jn[j] = (sel != nullptr && col < p.topk) ? sel[col] : -1;
      }
    };
    if (tile_begin >= 1 && tile_begin < tile_end) load_sel(tile_begin);
    int last_it[4] = {-1, -1, -1, -1};  // the last tile whose pair g was issued
    bool ok = true;
    for (int tile = tile_begin; tile < tile_end && ok; ++tile) {
      const int it = tile - tile_begin;
      int rc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = 4 * lane + j;
        int64_t src = -1;
        if (tile == 0) {
          const int64_t pos = lo_eff + r;
          if (pos <= t && r < p.window) {
            if (t - lo_eff + 1 > win_cap) set_flag(p.flags, CSA2_FLAG_BAD_WINDOW);
            else src = win_b0 + (pos % win_cap);
          }
        } else {
          // entries outside this launch's shard of the pool are not its rows
          const int32_t jj = jn[j];
          if (jj >= 0 && jj >= p.shard_lo && jj < p.shard_hi) {
            const int64_t jr = (int64_t)jj - p.shard_lo;
            if (jr < plen) src = pool_b0 + jr;
            else set_flag(p.flags, CSA2_FLAG_BAD_TOPK_INDEX);
          } else if (jj < -1) {
            set_flag(p.flags, CSA2_FLAG_BAD_TOPK_INDEX);
          }
        }
        if (src > 0x7FFFFFFFll) {  // beyond a tensor coordinate: not a row of any real buffer
          set_flag(p.flags, tile == 0 ? CSA2_FLAG_BAD_WINDOW : CSA2_FLAG_BAD_TOPK_INDEX);
          src = -1;
        }
        rc[j] = (int)src;
      }
      // row masks for the math warps, published before this tile's arrivals
      uint32_t mw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) mw[j] = __ballot_sync(0xffffffffu, rc[j] >= 0);
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) mask[(it & 1) * 4 + j] = mw[j];
      }
      const CUtensorMap* map = tile == 0 ? &win_map : &pool_map;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        // pair g still holds the previous tile's rows until its PV block is done
        if (it > 0) ok = mbar_wait(base_s + TB_EMPTY + 8 * g, (uint32_t)((it - 1) & 1), p.flags);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) mbar_expect_tx(base_s + TB_FULL + 8 * g, kPairBytes);
        __syncwarp();
#pragma unroll
        for (int cb = 2 * g; cb < 2 * g + 2; ++cb)
          tma_gather4(base_s + SM_KV + (uint32_t)cb * 16384u + (uint32_t)lane * 512u, map,
                      base_s + TB_FULL + 8 * g, 64 * cb, rc[0], rc[1], rc[2], rc[3]);
        last_it[g] = it;
      }
      // the next tile's entries are in flight while this tile is processed
      if (ok && tile + 1 < tile_end) load_sel(tile + 1);
    }
    // no copy may still be landing when the CTA exits
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (last_it[g] >= 0) mbar_wait(base_s + TB_FULL + 8 * g, (uint32_t)(last_it[g] & 1), p.flags, 1000000000ull);
  } else {
    // ---------------- math warps (thread 0 also issues the tensor-core work)
    const SyncMath sy;
    float lsum[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) lsum[k] = 0.f;
    uint32_t sphase = 0;
    bool aborted = false;
    // Q landed; its rope channels split into hi + lo before the first product
    cp_async_wait_all();
    sy.sync();
    if (p.rp.pairs > 0 && tile_begin < tile_end) q_rope_split(sm, p.rp);
    fence_proxy_async_smem();  // Q's generic-proxy writes, before the tensor cores read them
    sy.sync();
    const int n_ks = p.rp.pairs > 0 ? 36 : 32;
    for (int tile = tile_begin; tile < tile_end; ++tile) {
      const int it = tile - tile_begin;
      bool ok = true;
      if (tid == 0) {
        // S^T = KV . Q^T: K steps 8g .. 8g+7 read channel pair g as it lands;
        // steps 32..35 add the rope residual block of q against the last block
        tc_fence_after();
#pragma unroll 1
        for (int g = 0; g < 4 && ok; ++g) {
          ok = mbar_wait(base_s + TB_FULL + 8 * g, (uint32_t)(it & 1), p.flags);
          if (!ok) break;
          const int ks1 = g == 3 ? n_ks : 8 * g + 8;
#pragma unroll 4
          for (int ks = 8 * g; ks < ks1; ++ks) {
            const uint32_t koff = (uint32_t)(ks & 3) * 32u;
            const uint32_t kblk = ks < 32 ? (uint32_t)(ks >> 2) : 7u;
            const uint64_t ad = sdesc_sw128(base_s + SM_KV + kblk * 16384u + koff, 16u, 1024u);
            const uint64_t bd = sdesc_sw128(base_s + SM_Q + (uint32_t)(ks >> 2) * 8192u + koff, 16u, 1024u);
            mma_bf16_ss(tmem_s, ad, bd, kIdescQK, ks > 0 ? 1u : 0u);
          }
        }
        mma_commit(s_bar);
      }
      ok = mbar_wait(s_bar, sphase, p.flags) && ok;
      sphase ^= 1u;
      if (!sy.all(ok)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      // this tile's row masks (the phase is complete: thread 0 waited for it)
      mbar_wait(base_s + TB_FULL + 24, (uint32_t)(it & 1), p.flags);
      const bool valid = ((mask[(it & 1) * 4 + (row & 3)] >> (row >> 2)) & 1u) != 0;
      tile_softmax(p, sm, tmem_s, tmem_o, lane_base, valid, tile == tile_begin, &misc[3], lsum, sy);
      // O^T += KV^T . P^T in four blocks of 128 output dims; block mt reads
      // channel pair mt only, and its commit lets the producer refill it
      if (tid == 0) {
        tc_fence_after();
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad = sdesc_sw128(base_s + SM_KV + (uint32_t)(2 * mt) * 16384u + (uint32_t)ks * 2048u,
                                            16384u, 1024u);
            const uint64_t bd = sdesc_sw128(base_s + SM_P + (uint32_t)ks * 2048u, 8192u, 1024u);
            mma_bf16_ss(tmem_o + 64u * (uint32_t)mt, ad, bd, kIdescPV, (tile > tile_begin || ks > 0) ? 1u : 0u);
          }
          mma_commit(base_s + TB_EMPTY + 8 * mt);
        }
      }
    }
    // every tensor-core operation issued has completed before O^T is read or
    // its memory freed (after a timeout: the phase given up on, then this one)
    if (tid == 0) mma_commit(s_bar);
    bool done;
    if (!aborted) {
      done = mbar_wait(s_bar, sphase, p.flags);
    } else {
      mbar_wait(s_bar, sphase ^ 1u, p.flags, 1000000000ull);
      done = mbar_wait(s_bar, sphase, p.flags, 1000000000ull);
    }
    done = sy.all(done);
    tc_fence_after();
    const bool have_o = (tile_begin < tile_end) && !aborted && done;
    attend_store(p, sm, qi, split, have_o, lsum, tmem_o, lane_base, sink_l2, sy);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, kTmemCols);
}

// ---------------------------------------------------------------- host side

typedef CUresult (*TensorMapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static TensorMapEncodeFn tensor_map_encoder() {
  static TensorMapEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TensorMapEncodeFn>(f);
  });
  return fn;
}

// A [rows, 512] bf16 row buffer as a gather source: boxes of 64 channels x 1
// row (4 rows a gather4), 128-byte swizzle. The row extent is the largest
// tensor coordinate: the kernel checks every row it reads against the
// caller's offsets, as the thread-gathered kernel does. A NULL buffer (never
// read) gets an all-zero map.
static cudaError_t rows_map(const void* base, CUtensorMap* m) {
  std::memset(m, 0, sizeof(*m));
  if (base == nullptr) return cudaSuccess;
  const TensorMapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {(cuuint64_t)kDim, (cuuint64_t)0x7FFFFFFF};
  const cuuint64_t gstr[1] = {(cuuint64_t)kDim * 2};
  const cuuint32_t box[2] = {64, 1};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstr, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_attend_tiles_tma(cudaStream_t st, const AttendParams& p, int* n_launch) {
  alignas(64) CUtensorMap win_map, pool_map;
  cudaError_t e = rows_map(p.win_kv, &win_map);
  if (e == cudaSuccess) e = rows_map(p.topk_idx != nullptr ? p.pool_kv : nullptr, &pool_map);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attend_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(p.n_query * p.n_split));
  e = launch_ex(attend_tma_kernel, grid, dim3(kTmaThreads), kAttSmemBytes, st, p.pdl != 0, p.priority, p, win_map,
                pool_map);
  if (e != cudaSuccess) return e;
  *n_launch += 1;
  return cudaGetLastError();
}

}  // namespace csa2
