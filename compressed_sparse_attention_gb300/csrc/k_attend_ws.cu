// Two-source sparse attention for bf16 rows, warp-specialised ("Reading Notes
// of DeepSeek-V4.1-Flash", section 3a and section 3f, C2 step 3; the
// products, the softmax and the epilogue are those of attend_tile.cuh,
// shared with the thread-gathered kernel of k_attend.cu).
//
// A CTA holds 8 math warps and 4 producer warps. The first tile of a CTA has
// nothing to overlap with: the math warps gather it themselves, all 256
// threads, as the thread-gathered kernel does. For every later tile the
// producers compute the 128 row sources (thread p: row p) and gather the rows
// with 16-byte cp.async into the 128-byte-swizzled operand layout (a missing
// row reads zeros). A tile lands as four pairs of 64-channel blocks, all four
// in flight at once; for each pair every producer thread waits for its own
// copies, fences them into the async proxy and arrives on the pair's barrier
// full[g] (128 arrivals). Thread 0 of the math warps issues the pair's QK^T
// steps as soon as it completes.
// The PV product of tile i runs as four blocks of 128 output dims. Block g
// reads only channel pair g, and its tcgen05.commit arrives on empty[g], so
// the producers refill pair g with tile i+1's rows while blocks g+1..3 still
// run. The gather of the next tile thereby overlaps this tile's PV product
// and the next tile's QK^T product, and the math warps never wait on a copy
// they issued. The row sources double as the math warps' row masks; they are
// written before the producers' arrivals and read after full[3] completes.
// Every mbarrier wait is bounded: on a timeout the waiter records
// CSA2_FLAG_WAIT_TIMEOUT, the warps agree (barrier reductions) to stop, and
// what is in flight lands before tensor memory is freed.
//
// Gathering with the tensor memory accelerator instead (tile::gather4, 4 rows
// of 128 B an instruction) was built and measured: one warp issuing a tile's
// 256 instructions took 8.5 us a tile, four warps 3.0 us, against 2.2 us for
// cp.async from 256 threads on random rows of a 512 MiB buffer (1.3 us
// against 2.3 us from L2). The instructions' issue rate, not the copy engine,
// bounds it.
#include "attend_tile.cuh"

namespace csa2 {

constexpr int kProdWarps = 4;
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kWsThreads = kAttThreads + kProdThreads;
// past the shared layout of attend_tile.cuh: row sources and barriers
constexpr uint32_t WS_ROWS = SM_TOTAL;          // int32 [2][128] row of each tile row, -1: none
constexpr uint32_t WS_S = WS_ROWS + 1024;       // S^T ready, or all tensor-core work done
constexpr uint32_t WS_FULL = WS_S + 8;          // [4] channel pair g of the tile landed
constexpr uint32_t WS_EMPTY = WS_FULL + 32;     // [4] PV block g done: pair g may be refilled
constexpr uint32_t kWsSmemBytes = WS_EMPTY + 32 + 1024;  // + alignment slack
static_assert(kWsSmemBytes <= 232448, "shared memory of one CTA");

// barriers of the 128 producer threads (named barrier 2)
__device__ __forceinline__ void prod_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ bool prod_all(bool v) {
  uint32_t r;
  asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 2, 128, p;\nselp.u32 %0, 1, 0, q;\n}"
               : "=r"(r)
               : "r"((uint32_t)v)
               : "memory");
  return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__global__ void __launch_bounds__(kWsThreads, 1) attend_ws_kernel(const AttendParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_s - raw_s);
  float* m_run = reinterpret_cast<float*>(sm + SM_MRUN);
  float* l_run = reinterpret_cast<float*>(sm + SM_LRUN);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + SM_MISC);  // [2] tmem slot, [3] rescale
  int32_t* rows = reinterpret_cast<int32_t*>(sm + WS_ROWS);
  const uint32_t s_bar = base_s + WS_S;
  const uint32_t tslot = base_s + SM_MISC + 8;

  if (p.pdl) pdl_trigger();  // the merge may take the room this grid leaves
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp >= kAttWarps;
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
    cp_async_commit();
  }
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
      mbar_init(base_s + WS_FULL + 8 * g, kProdThreads);
      mbar_init(base_s + WS_EMPTY + 8 * g, 1);
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
  const int64_t lo_eff = max(max((int64_t)0, lo_raw), t - (int64_t)p.window + 1);
  const int64_t plen = q_ok ? (pool_b1 - pool_b0) : 0;
  const int32_t* sel = p.topk_idx != nullptr ? p.topk_idx + (int64_t)qi * p.topk : nullptr;
  // selection entry of row r of selected tile `tile` (-1 past k)
  auto sel_at = [&](int tile, int r) -> int32_t {
    const int col = (tile - 1) * kTileRows + r;
    return (sel != nullptr && col < p.topk) ? sel[col] : -1;
  };
  // source row of tile row r (window tile: window position; selected tile:
  // entry j of the selection), -1 for none; bad entries are recorded
  auto row_source = [&](int tile, int r, int32_t j) -> int32_t {
    int64_t src = -1;
    if (tile == 0) {
      const int64_t pos = lo_eff + r;
      if (pos <= t && r < p.window) {
        if (t - lo_eff + 1 > win_cap) set_flag(p.flags, CSA2_FLAG_BAD_WINDOW);
        else src = win_b0 + (pos % win_cap);
      }
    } else if (j >= 0 && j >= p.shard_lo && j < p.shard_hi) {
      // entries outside this launch's shard of the pool are not its rows
      const int64_t jr = (int64_t)j - p.shard_lo;
      if (jr < plen) src = pool_b0 + jr;
      else set_flag(p.flags, CSA2_FLAG_BAD_TOPK_INDEX);
    } else if (j < -1) {
      set_flag(p.flags, CSA2_FLAG_BAD_TOPK_INDEX);
    }
    if (src > 0x7FFFFFFFll) {  // not a row of any buffer that fits in memory
      set_flag(p.flags, tile == 0 ? CSA2_FLAG_BAD_WINDOW : CSA2_FLAG_BAD_TOPK_INDEX);
      src = -1;
    }
    return (int32_t)src;
  };

  if (producer) {
    // ---------------- producer warps: the second and later tiles
    const int pt = tid - kAttThreads;  // 0 .. 127: this thread's row of each tile
    // Launched programmatically after the step's top-k, the first read of the
    // selection waits for it (a plain launch returns at once).
    int32_t jn = -1;
    if (tile_begin + 1 < tile_end) {
      pdl_wait();
      jn = sel_at(tile_begin + 1, pt);
    }
    bool ok = true;
    for (int tile = tile_begin + 1; tile < tile_end && ok; ++tile) {
      const int it = tile - tile_begin;
      int32_t* rows_t = rows + (it & 1) * kTileRows;
      rows_t[pt] = row_source(tile, pt, jn);
      if (tile + 1 < tile_end) jn = sel_at(tile + 1, pt);  // in flight while this tile is gathered
      prod_sync();  // every row source of this tile is in place
      const uint16_t* kv = reinterpret_cast<const uint16_t*>(p.pool_kv);
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        // pair g holds the previous tile's rows until its PV block is done
        ok = prod_all(mbar_wait(base_s + WS_EMPTY + 8 * g, (uint32_t)((it - 1) & 1), p.flags));
        if (!ok) break;
        // 16 chunks of 16 B a row for the pair; a half warp copies one row's 256 B
#pragma unroll
        for (int u = 0; u < kTileRows * 16 / kProdThreads; ++u) {
          const int i = pt + kProdThreads * u;
          const int r = i >> 4;
          const int c = 16 * g + (i & 15);
          const int32_t s = rows_t[r];
          const uint32_t dst = base_s + SM_KV + (uint32_t)(c >> 3) * 16384u + (uint32_t)r * 128u +
                               ((uint32_t)((c & 7) ^ (r & 7)) << 4);
          const uint16_t* gp = s >= 0 ? kv + (int64_t)s * kDim + 8 * c : kv;
          cp_async16(dst, gp, s >= 0 ? 16u : 0u);
        }
        cp_async_commit();
      }
      if (!ok) break;
      // each pair goes to the tensor cores once this thread's copies of it
      // have landed, fenced into the async proxy (all four are in flight)
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        cp_async_wait_pending(3 - g);
        fence_proxy_async_smem();
        mbar_arrive(base_s + WS_FULL + 8 * g);
      }
    }
    cp_async_wait_all();  // no copy may still be landing when the CTA exits
  } else {
    // ---------------- math warps (thread 0 also issues the tensor-core work)
    const SyncMath sy;
    float lsum[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) lsum[k] = 0.f;
    uint32_t sphase = 0;
    bool aborted = false;
    const int n_ks = p.rp.pairs > 0 ? 36 : 32;
    // S^T = KV . Q^T for channel pair g: K steps 8g .. 8g+7, and for the last
    // pair steps 32..35, which add the rope residual block of q against the
    // last channel block (thread 0)
    auto issue_qk = [&](int g) {
      const int ks1 = g == 3 ? n_ks : 8 * g + 8;
#pragma unroll 4
      for (int ks = 8 * g; ks < ks1; ++ks) {
        const uint32_t koff = (uint32_t)(ks & 3) * 32u;
        const uint32_t kblk = ks < 32 ? (uint32_t)(ks >> 2) : 7u;
        const uint64_t ad = sdesc_sw128(base_s + SM_KV + kblk * 16384u + koff, 16u, 1024u);
        const uint64_t bd = sdesc_sw128(base_s + SM_Q + (uint32_t)(ks >> 2) * 8192u + koff, 16u, 1024u);
        mma_bf16_ss(tmem_s, ad, bd, kIdescQK, ks > 0 ? 1u : 0u);
      }
    };
    if (tile_begin < tile_end) {
      // The first tile has nothing to overlap with: the math warps gather it
      // themselves, in four commit groups (one per channel pair) behind Q's,
      // and issue each pair's QK^T steps as it lands. A CTA whose first tile
      // is selected waits for the step's top-k first.
      if (tid < kTileRows) {
        int32_t j = -1;
        if (tile_begin >= 1) {
          pdl_wait();
          j = sel_at(tile_begin, tid);
        }
        rows[tid] = row_source(tile_begin, tid, j);
      }
      sy.sync();
      const uint16_t* kv = reinterpret_cast<const uint16_t*>(tile_begin == 0 ? p.win_kv : p.pool_kv);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
#pragma unroll
        for (int u = 0; u < kTileRows * 16 / kAttThreads; ++u) {
          const int i = tid + kAttThreads * u;
          const int r = i >> 4;
          const int c = 16 * g + (i & 15);
          const int32_t s = rows[r];
          const uint32_t dst = base_s + SM_KV + (uint32_t)(c >> 3) * 16384u + (uint32_t)r * 128u +
                               ((uint32_t)((c & 7) ^ (r & 7)) << 4);
          const uint16_t* gp = s >= 0 ? kv + (int64_t)s * kDim + 8 * c : kv;
          cp_async16(dst, gp, s >= 0 ? 16u : 0u);
        }
        cp_async_commit();
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        cp_async_wait_pending(3 - g);
        if (g == 0 && p.rp.pairs > 0) {
          sy.sync();  // Q complete: its rope channels split into hi + lo
          q_rope_split(sm, p.rp);
        }
        fence_proxy_async_smem();  // generic-proxy writes, before the tensor cores read them
        sy.sync();
        if (tid == 0) {
          tc_fence_after();
          issue_qk(g);
        }
      }
      if (tid == 0) mma_commit(s_bar);
    } else {
      cp_async_wait_all();  // a query without tiles: no copy of Q may still be landing
    }
    for (int tile = tile_begin; tile < tile_end; ++tile) {
      const int it = tile - tile_begin;
      bool ok = true;
      if (it > 0 && tid == 0) {
        // later tiles: each pair's steps as the producers hand it over
        tc_fence_after();
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          ok = mbar_wait(base_s + WS_FULL + 8 * g, (uint32_t)((it - 1) & 1), p.flags);
          if (!ok) break;
          issue_qk(g);
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
      // this tile's row sources (for a later tile: the phase is complete,
      // thread 0 waited for it)
      if (it > 0) mbar_wait(base_s + WS_FULL + 24, (uint32_t)((it - 1) & 1), p.flags);
      const bool valid = rows[(it & 1) * kTileRows + row] >= 0;
      tile_softmax(p, sm, tmem_s, tmem_o, lane_base, valid, tile == tile_begin, &misc[3], lsum, sy);
      // O^T += KV^T . P^T in four blocks of 128 output dims; block mt reads
      // channel pair mt only, and its commit lets the producers refill it
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
          mma_commit(base_s + WS_EMPTY + 8 * mt);
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

cudaError_t launch_attend_tiles_ws(cudaStream_t st, const AttendParams& p, int* n_launch) {
  cudaError_t e = cudaFuncSetAttribute(attend_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kWsSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(p.n_query * p.n_split));
  e = launch_ex(attend_ws_kernel, grid, dim3(kWsThreads), kWsSmemBytes, st, p.pdl != 0, p.priority, p);
  if (e != cudaSuccess) return e;
  *n_launch += 1;
  return cudaGetLastError();
}

}  // namespace csa2
