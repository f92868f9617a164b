// Two-source sparse attention with a per-head sink ("Reading Notes of
// DeepSeek-V4.1-Flash", section 3a and section 3f, C2 step 3; "DeepSeek-V4.1-
// Flash on WASTE", "What is new" item 1: the sink enters the denominator only,
// the output's rope channels are rotated back by -t).
//
// One CTA owns one query and a contiguous range of 128-row tiles: tile 0 is
// the query's window, tiles 1.. are the selected compressed entries, 128 per
// tile (the products, layout and softmax are those of attend_tile.cuh). In
// this file the CTA's threads gather the rows themselves, which lets them
// convert fp8 and fp4 rows to bf16 on the way. With several CTAs per
// query (split-K) each writes its unnormalised O^T and (max, sum) and a merge
// kernel combines them with the sink.
#include "attend_tile.cuh"

namespace csa2 {

// KVF: 0 bf16 rows; 1 fp8 rows; 2 fp8 window rows and fp4 pool rows
template <int KVF>
__global__ void __launch_bounds__(kAttThreads, 1) attend_kernel(const AttendParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_s - raw_s);
  float* m_run = reinterpret_cast<float*>(sm + SM_MRUN);
  float* l_run = reinterpret_cast<float*>(sm + SM_LRUN);
  int64_t* rows = reinterpret_cast<int64_t*>(sm + SM_ROWS);
  // misc: [0..1] mbar, [2] tmem slot, [3] rescale, [4] abort, [5..7] the shard's selection columns (first, last, count)
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + SM_MISC);
  const uint32_t mbar = base_s + SM_MISC;
  const uint32_t tslot = base_s + SM_MISC + 8;

  if (p.pdl) pdl_trigger();  // the merge may take the room this grid leaves
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;                  // lane quadrant
  const int row = quad * 32 + lane;           // this thread's tile row / output dim in a 128 block
  // CTAs are numbered split-major (all queries' first CTAs first, which hold
  // the window tile and start before the selection exists). Split 0 takes
  // the launch's first lead_tiles tiles, the others tiles_per_split each.
  const int qi = blockIdx.x % p.n_query, split = blockIdx.x / p.n_query;
  const int lead = p.lead_tiles;
  const int tile_begin = split == 0 ? p.tile_base : p.tile_base + lead + (split - 1) * p.tiles_per_split;
  const int tile_cap0 = split == 0 ? tile_begin + lead : tile_begin + p.tiles_per_split;
  const int tile_cap = min(tile_cap0, p.tile_base + p.tile_count);
  // every load that depends only on the query index is issued before the
  // setup below, so that their latencies overlap: the query's position and
  // sequence, Q itself, and (after the wait below) this thread's first
  // selection entry
  const int64_t t = p.q_pos[qi];
  const int b = p.seq_of_q[qi];
  // selection entry of this thread's row in selected tile `tile` (-1 past
  // the columns [sel_off, sel_lim) the selected tiles take)
  int sel_off = 0, sel_lim = p.topk;
  auto sel_entry = [&](int tile, int tile_lim) -> int32_t {
    const int col = sel_off + (tile - 1) * kTileRows + tid;
    return (tid < kTileRows && tile >= 1 && tile < tile_lim && col < sel_lim && p.topk_idx != nullptr)
               ? p.topk_idx[(int64_t)qi * p.topk + col]
               : -1;
  };
  // A plain launch fetches this thread's first selection entry at once; a
  // programmatic one (after the step's top-k) only after pdl_wait() below.
  int32_t j_next = p.pdl ? -1 : sel_entry(tile_begin, tile_cap);
  // Q is copied asynchronously into its swizzled K-major slots (it lands
  // together with the first tile's rows); the rope channels are rotated in
  // place once both have arrived
  if (tile_begin < tile_cap) copy_q_async(p, base_s, qi);
  cp_async_commit();  // Q's group lands before any KV group of the first tile
  const bool q_ok = (b >= 0 && b < p.n_seq && t >= 0);
  int tile_end = q_ok ? tile_cap : tile_begin;
  if (!q_ok && tid == 0 && split == 0) set_flag(p.flags, CSA2_FLAG_BAD_QUERY);
  const int bs = q_ok ? b : 0;  // offsets of a valid sequence (unused when !q_ok)
  const QueryRows qr = query_rows(p, t, bs, q_ok);
  // Launched programmatically after the step's top-k, this CTA may run before
  // the selection exists: everything above reads step inputs only, the window
  // tile needs no selection, and the selection is read after pdl_wait()
  // before the first selected tile (a plain launch returns at once).
  // Deferred only when the selection may still be in the making and the
  // query's first CTA has the window tile to run meanwhile (several CTAs a
  // query); otherwise the first tile's entries are fetched now, ahead of it.
  const bool defer_sel = p.pdl != 0 && p.n_split > 1;
  bool sel_ready = !defer_sel;
  if (p.pdl && sel_ready) {
    pdl_wait();
    j_next = sel_entry(tile_begin, tile_cap);
  }

  if (warp == 0) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(mbar, 1);
    fence_mbar_init();
    misc[3] = 0;
    misc[4] = 0;
    misc[5] = 0xFFFFFFFFu;
    misc[6] = 0u;
    misc[7] = 0u;
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
  bool q_pending = true;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = misc[2];
  const uint32_t tmem_s = taddr;        // columns [0, 64)
  const uint32_t tmem_o = taddr + 64;   // columns [64, 320)
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  uint32_t phase = 0;
  bool aborted = false;

  // One shard's part (csa2_attend_partial): when the selection's entries in
  // the shard fill one run of columns (a selection in ascending order, as
  // csa2_topk and csa2_topk_merge write it), the selected tiles take that run
  // only, 128 entries a tile; otherwise every column, the others skipped row
  // by row. A shard holding a G-th of the pool then runs about k / G rows
  // instead of k.
  if (p.direct == 2 && p.topk_idx != nullptr && q_ok) {
    uint32_t first = 0xFFFFFFFFu, last = 0u, cnt = 0u;
    for (int c = tid; c < p.topk; c += kAttThreads) {
      const int32_t j = p.topk_idx[(int64_t)qi * p.topk + c];
      if (j >= 0 && j >= p.shard_lo && j < p.shard_hi) {
        first = min(first, (uint32_t)c);
        last = max(last, (uint32_t)c);
        ++cnt;
      }
    }
    first = __reduce_min_sync(0xffffffffu, first);
    last = __reduce_max_sync(0xffffffffu, last);
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0 && cnt > 0) {
      atomicMin(&misc[5], first);
      atomicMax(&misc[6], last);
      atomicAdd(&misc[7], cnt);
    }
    __syncthreads();
    const uint32_t n_in = misc[7];
    if (n_in == 0u || misc[6] - misc[5] + 1u == n_in) {
      sel_off = n_in == 0u ? 0 : (int)misc[5];
      sel_lim = sel_off + (int)n_in;
      tile_end = min(tile_end, 1 + ((int)n_in + kTileRows - 1) / kTileRows);
      if (tile_end < tile_begin) tile_end = tile_begin;
      j_next = sel_entry(tile_begin, tile_end);
    }
  }

  // Two passes over the tiles: with the selection deferred, a CTA that starts
  // at the window tile runs it alone in the first pass and waits for the
  // selection between the passes (a wait inside the tile loop measured 4 %
  // slower in prefill, where it never runs); otherwise the first pass takes
  // every tile.
  if (defer_sel && tile_begin >= 1) {
    pdl_wait();
    j_next = sel_entry(tile_begin, tile_end);
    sel_ready = true;
  }
  float lsum[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) lsum[k] = 0.f;
  int tile = tile_begin;
  for (int pass = 0; pass < 2; ++pass) {
  const int pass_end = (pass == 0 && !sel_ready) ? min(tile_end, 1) : tile_end;
  if (pass == 1 && !sel_ready && tile < tile_end) {
    pdl_wait();
    j_next = sel_entry(tile, tile_end);
    sel_ready = true;
  }
  for (; tile < pass_end && !aborted; ++tile) {
    // ---- row sources of this tile (one thread per row, the first 128)
    if (tid < kTileRows) {
      const int32_t j_cur = j_next;
      j_next = sel_ready ? sel_entry(tile + 1, tile_end) : -1;  // one tile ahead
      rows[tid] = tile_row_src(p, qr, tile, tid, j_cur);
    }
    __syncthreads();
    // ---- gather the tile's rows into the swizzled KV operand
    const void* kvsrc = (tile == 0) ? p.win_kv : p.pool_kv;
    if constexpr (KVF == 0) {
      gather_bf16_tile(base_s, rows, reinterpret_cast<const uint16_t*>(kvsrc));
    } else if (KVF == 2 && tile != 0) {
      // fp4 pool rows: 256 B of E2M1 codes + 32 e4m3 scales; lane l converts
      // channels 16l .. 16l+15 (8 code bytes, scale l), 8 rows' loads in flight
      const uint8_t* kv = reinterpret_cast<const uint8_t*>(p.pool_kv);
      constexpr int kBatch = 8;
#pragma unroll 1
      for (int r0 = warp; r0 < kTileRows; r0 += kAttWarps * kBatch) {
        uint2 codes[kBatch];
        uint8_t sb[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int64_t src = rows[r0 + kAttWarps * j];
          codes[j] = make_uint2(0u, 0u);
          sb[j] = 0;
          if (src >= 0) {
            codes[j] = ldg_stream8(kv + src * (kDim / 2) + 8 * lane);
            sb[j] = p.pool_scale[src * (kDim / 16) + lane];
          }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int r = r0 + kAttWarps * j;
          const float sc = e4m3_value(sb[j]) * kE2M1Unscale;  // code values arrive scaled by 2^-14
          uint32_t o[8];
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const uint32_t w = ((b < 4 ? codes[j].x : codes[j].y) >> (8 * (b & 3))) & 0xFFu;
            const float2 f = e2m1x2_to_float2_scaled(w);
            o[b] = pack_bf16(f.x * sc, f.y * sc);  // exact: <= 6 significant bits
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * lane + cc;  // bf16 chunk: channels 8c .. 8c+7
            const uint32_t off = SM_KV + (uint32_t)(c >> 3) * 16384u + (uint32_t)r * 128u +
                                 ((uint32_t)((c & 7) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(sm + off) = make_uint4(o[4 * cc], o[4 * cc + 1], o[4 * cc + 2], o[4 * cc + 3]);
          }
        }
      }
    } else {
      const uint8_t* kv = reinterpret_cast<const uint8_t*>(kvsrc);
      const uint8_t* ksc = (tile == 0) ? p.win_scale : p.pool_scale;
      // a warp takes rows warp, warp+8, ...; the loads of 8 rows are in
      // flight together before any of them is converted
      constexpr int kBatch = 8;
#pragma unroll 1
      for (int r0 = warp; r0 < kTileRows; r0 += kAttWarps * kBatch) {
        uint4 codes[kBatch];
        uint8_t sb[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int64_t src = rows[r0 + kAttWarps * j];
          codes[j] = make_uint4(0u, 0u, 0u, 0u);
          sb[j] = 0;
          if (src >= 0) {
            codes[j] = ldg_stream16(kv + src * kDim + 16 * lane);
            sb[j] = ksc[src * (kDim / 32) + (lane >> 1)];
          }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int r = r0 + kAttWarps * j;
          const float sc = ue8m0_value(sb[j]);
          const uint32_t cw[4] = {codes[j].x, codes[j].y, codes[j].z, codes[j].w};
          uint32_t o[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 a = e4m3x2_to_float2((uint16_t)(cw[k] & 0xFFFFu));
            const float2 c2 = e4m3x2_to_float2((uint16_t)(cw[k] >> 16));
            o[2 * k] = pack_bf16(a.x * sc, a.y * sc);
            o[2 * k + 1] = pack_bf16(c2.x * sc, c2.y * sc);
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * lane + cc;  // bf16 chunk: channels 8c .. 8c+7
            const uint32_t off = SM_KV + (uint32_t)(c >> 3) * 16384u + (uint32_t)r * 128u +
                                 ((uint32_t)((c & 7) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(sm + off) = make_uint4(o[4 * cc], o[4 * cc + 1], o[4 * cc + 2], o[4 * cc + 3]);
          }
        }
      }
    }
    // bf16 tiles arrive in kKvGroups commit groups and their QK^T steps are
    // issued group by group; the converting gathers above are complete
    constexpr int n_groups = (KVF == 0) ? kKvGroups : 1;
    const int n_ks = p.rp.pairs > 0 ? 36 : 32;
#pragma unroll
    for (int g = 0; g < n_groups; ++g) {
      if constexpr (KVF == 0) cp_async_wait_pending(n_groups - 1 - g);
      else cp_async_wait_all();
      if (g == 0 && q_pending) {
        q_pending = false;
        if (p.rp.pairs > 0) {
          __syncthreads();
          q_rope_split(sm, p.rp);
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      // ---- S^T = KV . Q^T: K steps 0..31 cover the 8 channel blocks (this
      // group's share of them); 32..35 add the rope residual block of q
      // against the KV's last channel block (the rope channels)
      if (tid == 0) {
        tc_fence_after();
        issue_qk(base_s, tmem_s, g, n_groups, n_ks > 32);
        if (g == n_groups - 1) mma_commit(mbar);
      }
    }
    bool ok = mbar_wait(mbar, phase, p.flags);
    phase ^= 1u;
    if (!__syncthreads_and(ok)) { aborted = true; break; }
    tc_fence_after();
    // ---- softmax over this tile's rows; P^T and O^T ready afterwards
    tile_softmax(p, sm, tmem_s, tmem_o, lane_base, rows[row] >= 0, tile == tile_begin, &misc[3], lsum, SyncCta{});
    // ---- O^T += KV^T . P^T
    if (tid == 0) {
      tc_fence_after();
      issue_pv(base_s, tmem_o, tile > tile_begin);
      mma_commit(mbar);
    }
    ok = mbar_wait(mbar, phase, p.flags);
    phase ^= 1u;
    if (!__syncthreads_and(ok)) { aborted = true; break; }
    tc_fence_after();
  }
  }

  // ---- epilogue (no copy of Q may still be landing when the CTA exits,
  // e.g. for a query without tiles)
  cp_async_wait_all();
  __syncthreads();
  const bool have_o = (tile_begin < tile_end) && !aborted;
  attend_store(p, sm, qi, split, have_o, lsum, tmem_o, lane_base, sink_l2, SyncCta{});
  if (aborted) {
    // let any tensor-core work still in flight land before freeing its memory
    mbar_wait(mbar, phase ^ 1u, p.flags, 1000000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, kTmemCols);
}

// Many queries, bf16 rows (chunked prefill): one persistent CTA per SM takes
// queries blockIdx.x, blockIdx.x + gridDim.x, ... and runs each query's
// tiles start to finish as attend_kernel does, with the output written
// directly. Between queries nothing waits: once the last tile's S^T is
// ready the next query's Q is copied into the free Q buffer, and once its PV
// product is done the next query's window rows are gathered into the free
// KV buffer, both before this query's epilogue, which then runs while they
// land (the epilogue reads O^T; the next query's first QK^T writes S^T, and
// its first PV, which overwrites O^T, comes after the epilogue). Tensor
// memory, the barrier and the sink are set up once per CTA.
__global__ void __launch_bounds__(kAttThreads, 1) attend_persist_kernel(const AttendParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_s - raw_s);
  float* m_run = reinterpret_cast<float*>(sm + SM_MRUN);
  float* l_run = reinterpret_cast<float*>(sm + SM_LRUN);
  int64_t* rows = reinterpret_cast<int64_t*>(sm + SM_ROWS);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + SM_MISC);  // [0..1] mbar, [2] tmem slot, [3] rescale
  float2* rope_tab = reinterpret_cast<float2*>(sm + SM_ROPE);
  const uint32_t mbar = base_s + SM_MISC;
  const uint32_t tslot = base_s + SM_MISC + 8;
  const uint16_t* win_kv = reinterpret_cast<const uint16_t*>(p.win_kv);
  const uint16_t* pool_kv = reinterpret_cast<const uint16_t*>(p.pool_kv);

  if (p.pdl) pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;
  if (warp == 0) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(mbar, 1);
    fence_mbar_init();
    misc[3] = 0;
  }
  const float sink_l2 = (tid < kHeads) ? p.sink[tid] * 1.4426950408889634f : 0.f;
  const bool rope = p.rp.pairs > 0;
  // the selection may be the previous kernel's output (csa2_step's top-k)
  if (p.pdl) pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = misc[2];
  const uint32_t tmem_s = taddr;        // columns [0, 64)
  const uint32_t tmem_o = taddr + 64;   // columns [64, 320)
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  uint32_t phase = 0;
  bool aborted = false;

  // query qi's position, sequence check, row layout and rope table row
  QueryRows qr{};
  bool q_ok = false;
  auto begin_query = [&](int qi) {
    const int64_t t = p.q_pos[qi];
    const int b = p.seq_of_q[qi];
    q_ok = (b >= 0 && b < p.n_seq && t >= 0);
    if (!q_ok && tid == 0) set_flag(p.flags, CSA2_FLAG_BAD_QUERY);
    qr = query_rows(p, t, q_ok ? b : 0, q_ok);
  };
  // the next query's Q (its own commit group) and window tile (four groups),
  // into buffers nothing reads any more
  auto prefetch_window = [&]() {
    if (tid < kTileRows) rows[tid] = q_ok ? tile_row_src(p, qr, 0, tid, -1) : -1;
    __syncthreads();
    gather_bf16_tile(base_s, rows, win_kv);
  };
  auto set_rope = [&]() {
    if (tid < p.rp.pairs) {
      float c = 1.f, sn = 0.f;
      if (q_ok) rope_cs(p.rp, tid, qr.t, c, sn);
      rope_tab[tid] = make_float2(c, sn);
    }
    if (tid < kHeads) {
      m_run[tid] = -INFINITY;
      l_run[tid] = 0.f;
    }
  };

  int qi = blockIdx.x;
  if (qi < p.n_query) {
    copy_q_async(p, base_s, qi);
    cp_async_commit();
    begin_query(qi);
    prefetch_window();
    set_rope();
  }
  while (qi < p.n_query) {
    const int qn = qi + (int)gridDim.x;
    const bool has_next = qn < p.n_query;
    const int n_t = q_ok ? p.n_tiles : 0;
    const int32_t* sel = p.topk_idx != nullptr ? p.topk_idx + (int64_t)qi * p.topk : nullptr;
    auto sel_at = [&](int tile) -> int32_t {
      const int col = (tile - 1) * kTileRows + tid;
      return (tid < kTileRows && tile >= 1 && tile < n_t && sel != nullptr && col < p.topk) ? sel[col] : -1;
    };
    float lsum[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) lsum[k] = 0.f;
    bool next_issued = false;
    for (int tile = 0; tile < n_t; ++tile) {
      const int32_t j_next = sel_at(tile + 1);  // in flight while this tile runs
#pragma unroll
      for (int g = 0; g < kKvGroups; ++g) {
        cp_async_wait_pending(kKvGroups - 1 - g);
        if (tile == 0 && g == 0 && rope) {
          __syncthreads();  // Q complete: its rope channels split into hi + lo
          q_rope_split(sm, p.rp);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
          tc_fence_after();
          issue_qk(base_s, tmem_s, g, kKvGroups, rope);
          if (g == kKvGroups - 1) mma_commit(mbar);
        }
      }
      bool ok = mbar_wait(mbar, phase, p.flags);
      phase ^= 1u;
      if (!__syncthreads_and(ok)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      if (tile == n_t - 1 && has_next) {
        copy_q_async(p, base_s, qn);  // every QK^T product of this query is done
        cp_async_commit();
      }
      tile_softmax(p, sm, tmem_s, tmem_o, lane_base, rows[row] >= 0, tile == 0, &misc[3], lsum, SyncCta{});
      if (tid == 0) {
        tc_fence_after();
        issue_pv(base_s, tmem_o, tile > 0);
        mma_commit(mbar);
      }
      ok = mbar_wait(mbar, phase, p.flags);
      phase ^= 1u;
      if (!__syncthreads_and(ok)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      if (tile + 1 < n_t) {
        if (tid < kTileRows) rows[tid] = tile_row_src(p, qr, tile + 1, tid, j_next);
        __syncthreads();
        gather_bf16_tile(base_s, rows, pool_kv);
      } else if (has_next) {
        begin_query(qn);
        prefetch_window();
        next_issued = true;
      }
    }
    if (aborted) break;
    if (has_next && !next_issued) {
      // a query without tiles: let its own copies land before reusing the buffers
      cp_async_wait_all();
      __syncthreads();
      copy_q_async(p, base_s, qn);
      cp_async_commit();
      begin_query(qn);
      prefetch_window();
    }
    __syncthreads();
    attend_store(p, sm, qi, 0, n_t > 0, lsum, tmem_o, lane_base, sink_l2, SyncCta{});
    // the epilogue's tensor-memory loads and its reads of the rope table and
    // the running (max, sum) are complete before the next query takes them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (has_next) set_rope();
    qi = qn;
  }
  cp_async_wait_all();  // no copy may still be landing when the CTA exits
  if (aborted) mbar_wait(mbar, phase ^ 1u, p.flags, 1000000000ull);  // tensor-core work in flight lands first
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, kTmemCols);
}

// merge of split-K partials: one CTA per (query, group of 4 heads); thread
// (head hl = tid/64, chunk = tid%64) owns channels 8*chunk .. 8*chunk+7. All
// splits' loads are issued before any is used.
constexpr int kMergeHeadsPerCta = 4;
__global__ void __launch_bounds__(256) attend_merge_kernel(const AttendParams p) {
  __shared__ float wsplit[8][kMergeHeadsPerCta];
  __shared__ float2 rope_tab[kMaxPairs];
  pdl_wait();  // the partials of the selected tiles (a plain launch returns at once)
  const int qi = blockIdx.x / (kHeads / kMergeHeadsPerCta);
  const int hg = blockIdx.x % (kHeads / kMergeHeadsPerCta);
  const int tid = threadIdx.x, hl = tid >> 6, chunk = tid & 63;
  const int h = hg * kMergeHeadsPerCta + hl;
  const int ns = p.n_slots;
  const float2* ml = p.ws_ml + (int64_t)qi * ns * kHeads;
  const int64_t t = p.q_pos[qi];
  // every load goes out before any is used: this thread's slices of the
  // partials (a split without rows may hold stale bytes; its weight is 0 and
  // its slice is never used) and, for the weight threads, the splits' (max, sum)
  const uint16_t* base = p.ws_o + ((int64_t)qi * ns * kHeads + h) * kDim + 8 * chunk;
  uint4 part[8];
#pragma unroll
  for (int s = 0; s < 8; ++s)
    part[s] = s < ns ? *reinterpret_cast<const uint4*>(base + (int64_t)s * kHeads * kDim) : make_uint4(0u, 0u, 0u, 0u);
  if (tid < kMergeHeadsPerCta) {
    const int hh = hg * kMergeHeadsPerCta + tid;
    float2 v[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) v[s] = s < ns ? ml[s * kHeads + hh] : make_float2(-INFINITY, 0.f);
    const float sk = p.sink[hh] * 1.4426950408889634f;
    float M = sk;
#pragma unroll
    for (int s = 0; s < 8; ++s) M = fmaxf(M, v[s].x);
    float den = 0.f;
    if (M != -INFINITY) {
      den = exp2f(sk - M);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (v[s].x != -INFINITY) den += v[s].y * exp2f(v[s].x - M);
    }
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s < ns) wsplit[s][tid] = (M == -INFINITY || v[s].x == -INFINITY) ? 0.f : exp2f(v[s].x - M) / den;
    if (p.lse) p.lse[(int64_t)qi * kHeads + hh] = (M == -INFINITY) ? -INFINITY : (M + log2f(den)) * 0.6931471805599453f;
  }
  if (tid >= 32 && tid - 32 < p.rp.pairs) {
    float c, sn;
    rope_cs(p.rp, tid - 32, t, c, sn);
    rope_tab[tid - 32] = make_float2(c, sn);
  }
  __syncthreads();
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    if (s < ns && wsplit[s][hl] != 0.f) {
      const float w = wsplit[s][hl];
      const uint32_t pw[4] = {part[s].x, part[s].y, part[s].z, part[s].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[2 * k] = fmaf(w, bf16lo(pw[k]), acc[2 * k]);
        acc[2 * k + 1] = fmaf(w, bf16hi(pw[k]), acc[2 * k + 1]);
      }
    }
  }
  const int first_rope = kDim - 2 * p.rp.pairs;
  if (p.rp.pairs > 0 && 8 * chunk >= first_rope) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 cs = rope_tab[(8 * chunk + 2 * k - first_rope) >> 1];
      const float x0 = acc[2 * k], x1 = acc[2 * k + 1];
      acc[2 * k] = x0 * cs.x + x1 * cs.y;       // rotation by -t
      acc[2 * k + 1] = x1 * cs.x - x0 * cs.y;
    }
  }
  uint4 o;
  o.x = pack_bf16(acc[0], acc[1]); o.y = pack_bf16(acc[2], acc[3]);
  o.z = pack_bf16(acc[4], acc[5]); o.w = pack_bf16(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(p.out + ((int64_t)qi * kHeads + h) * kDim + 8 * chunk) = o;
  // the next kernel (the next layer's compress in a decode loop) may launch
  // once every CTA is here; it still reads nothing before this grid is done
  pdl_trigger();
}

// Test aid for the bounded waits: one thread initialises an mbarrier that
// nothing ever arrives at and waits on its first phase with the attention
// kernels' own bounded wait; after limit_ns the wait gives up, records
// CSA2_FLAG_WAIT_TIMEOUT, and the kernel returns.
__global__ void wait_probe_kernel(uint32_t* flags, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
    mbar_wait(b, 0u, flags, limit_ns);
  }
}

cudaError_t launch_wait_probe(cudaStream_t st, uint32_t* flags, uint64_t limit_ns) {
  wait_probe_kernel<<<1, 32, 0, st>>>(flags, limit_ns);
  return cudaGetLastError();
}

// log-sum-exp combine of partials from several pool shards: one CTA per
// (query, 4 heads), thread (head hl = tid/64, chunk = tid%64) owning channels
// 8 chunk .. 8 chunk + 7. With M = max(max_g m_g, sink), the output is
// sum_g e^(m_g - M) O_g / (sum_g e^(m_g - M) l_g + e^(sink - M)), its rope
// channels rotated back by -t; lse = M + log(den).
constexpr int kCombineMaxParts = 16;
__global__ void __launch_bounds__(256) attend_combine_kernel(int n_query, int n_parts, const float* __restrict__ part_o,
                                                             const float* __restrict__ part_m,
                                                             const float* __restrict__ part_l,
                                                             const int64_t* __restrict__ q_pos,
                                                             const float* __restrict__ sink, const RopeParams rp,
                                                             uint16_t* __restrict__ out, float* __restrict__ lse) {
  __shared__ float wpart[kCombineMaxParts][kMergeHeadsPerCta];
  __shared__ float2 rope_tab[kMaxPairs];
  const int qi = blockIdx.x / (kHeads / kMergeHeadsPerCta);
  const int hg = blockIdx.x % (kHeads / kMergeHeadsPerCta);
  const int tid = threadIdx.x, hl = tid >> 6, chunk = tid & 63;
  const int h = hg * kMergeHeadsPerCta + hl;
  const int64_t t = q_pos[qi];
  // every load goes out before any is used: the weight threads' (m, l) of
  // all parts, and every thread's slices of the first four parts' O
  constexpr int kBatch = 4;
  float4 oa[kBatch], ob[kBatch];
  auto load_o = [&](int g0) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (g0 + u < n_parts) {
        const float4* src = reinterpret_cast<const float4*>(
            part_o + (((int64_t)(g0 + u) * n_query + qi) * kHeads + h) * kDim + 8 * chunk);
        oa[u] = src[0];
        ob[u] = src[1];
      }
    }
  };
  load_o(0);
  if (tid < kMergeHeadsPerCta) {
    const int hh = hg * kMergeHeadsPerCta + tid;
    float mv[kCombineMaxParts], lv[kCombineMaxParts];
#pragma unroll
    for (int g = 0; g < kCombineMaxParts; ++g) {
      mv[g] = g < n_parts ? part_m[((int64_t)g * n_query + qi) * kHeads + hh] : -INFINITY;
      lv[g] = g < n_parts ? part_l[((int64_t)g * n_query + qi) * kHeads + hh] : 0.f;
    }
    const float sk = sink[hh];
    float M = sk;
#pragma unroll
    for (int g = 0; g < kCombineMaxParts; ++g)
      if (g < n_parts) M = fmaxf(M, mv[g]);
    float den = 0.f;
    if (M != -INFINITY) {
      den = expf(sk - M);
#pragma unroll
      for (int g = 0; g < kCombineMaxParts; ++g)
        if (g < n_parts && mv[g] != -INFINITY) den += lv[g] * expf(mv[g] - M);
    }
#pragma unroll
    for (int g = 0; g < kCombineMaxParts; ++g)
      if (g < n_parts) wpart[g][tid] = (M == -INFINITY || mv[g] == -INFINITY) ? 0.f : expf(mv[g] - M) / den;
    if (lse) lse[(int64_t)qi * kHeads + hh] = (M == -INFINITY) ? -INFINITY : M + logf(den);
  }
  if (tid >= 32 && tid - 32 < rp.pairs) {
    float c, sn;
    rope_cs(rp, tid - 32, t, c, sn);
    rope_tab[tid - 32] = make_float2(c, sn);
  }
  __syncthreads();
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int g0 = 0; g0 < n_parts; g0 += kBatch) {
    if (g0 > 0) load_o(g0);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (g0 + u >= n_parts) break;
      const float w = wpart[g0 + u][hl];
      if (w == 0.f) continue;
      const float4 a = oa[u], b = ob[u];
      acc[0] = fmaf(w, a.x, acc[0]); acc[1] = fmaf(w, a.y, acc[1]);
      acc[2] = fmaf(w, a.z, acc[2]); acc[3] = fmaf(w, a.w, acc[3]);
      acc[4] = fmaf(w, b.x, acc[4]); acc[5] = fmaf(w, b.y, acc[5]);
      acc[6] = fmaf(w, b.z, acc[6]); acc[7] = fmaf(w, b.w, acc[7]);
    }
  }
  const int first_rope = kDim - 2 * rp.pairs;
  if (rp.pairs > 0 && 8 * chunk >= first_rope) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 cs = rope_tab[(8 * chunk + 2 * k - first_rope) >> 1];
      const float x0 = acc[2 * k], x1 = acc[2 * k + 1];
      acc[2 * k] = x0 * cs.x + x1 * cs.y;  // rotation by -t
      acc[2 * k + 1] = x1 * cs.x - x0 * cs.y;
    }
  }
  uint4 o;
  o.x = pack_bf16(acc[0], acc[1]); o.y = pack_bf16(acc[2], acc[3]);
  o.z = pack_bf16(acc[4], acc[5]); o.w = pack_bf16(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out + ((int64_t)qi * kHeads + h) * kDim + 8 * chunk) = o;
}

cudaError_t launch_attend_combine(cudaStream_t st, int n_query, int n_parts, const float* part_o, const float* part_m,
                                  const float* part_l, const int64_t* q_pos, const float* sink, const RopeParams& rp,
                                  uint16_t* out, float* lse, int* n_launch) {
  if (n_query == 0) return cudaSuccess;
  if (n_parts < 1 || n_parts > kCombineMaxParts) return cudaErrorInvalidValue;
  attend_combine_kernel<<<n_query * (kHeads / kMergeHeadsPerCta), 256, 0, st>>>(n_query, n_parts, part_o, part_m,
                                                                                part_l, q_pos, sink, rp, out, lse);
  *n_launch += 1;
  return cudaGetLastError();
}

int attend_num_tiles(int topk, bool has_idx) { return 1 + (has_idx ? (topk + kTileRows - 1) / kTileRows : 0); }

// How one attention call is cut, in one launch. With few queries (decode:
// 2 Q <= SMs) each query's tiles go to at most one wave of CTAs:
// floor(SMs / Q) CTAs a query (at most 8), the selected tiles split evenly
// (tps each) and the first CTA also taking the window tile, which needs no
// selection: launched after the step's top-k, it runs while the selection is
// still being made (or, see below, a CTA of its own takes the window tile). A merge combines the CTAs' partials. With many queries
// (prefill) one CTA per query runs every tile and writes the output directly.
AttendPlan attend_plan(int n_query, int topk, bool has_idx, int num_sms, bool own_window) {
  AttendPlan pl{};
  pl.n_tiles = attend_num_tiles(topk, has_idx);
  if (n_query < 1) n_query = 1;
  const int n_sel = pl.n_tiles - 1;
  int ns = 2 * n_query <= num_sms ? num_sms / n_query : 1;
  if (ns > n_sel) ns = n_sel;
  if (ns > 8) ns = 8;
  if (ns < 1) ns = 1;
  pl.ctas = num_sms;  // persistent CTAs of a one-CTA-a-query plan (one per SM)
  if (ns == 1) {
    pl.tps = pl.n_tiles;
    pl.lead = pl.n_tiles;
    pl.ns = 1;
    pl.n_slots = 0;
    return pl;
  }
  pl.tps = (n_sel + ns - 1) / ns;
  pl.ns = (n_sel + pl.tps - 1) / pl.tps;
  pl.lead = 1 + pl.tps;
  // own_window, with an SM to spare for every query: the window tile gets a
  // CTA of its own. After a short top-k the first CTA would otherwise still
  // be on the window tile when the selection is ready, and run its selected
  // tile after it (tiny decode 24.6 -> 22.0 us a step); after the long rows'
  // cluster top-k the window tile is long done, and a fifth partial only
  // lengthens the merge (1M decode +0.4 us).
  if (own_window && n_query * (pl.ns + 1) <= num_sms && pl.ns + 1 <= 8) {
    pl.lead = 1;
    pl.ns += 1;
  }
  pl.n_slots = pl.ns;
  return pl;
}

size_t attend_workspace_bytes(int n_query, const AttendPlan& pl) {
  if (pl.n_slots == 0) return 0;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)n_query * pl.n_slots * kHeads * kDim * 2) + al((size_t)n_query * pl.n_slots * kHeads * 8);
}

static void attach_ws(AttendParams& p, const AttendPlan& pl, void* ws) {
  p.n_slots = pl.n_slots;
  if (pl.n_slots > 0) {
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    p.ws_o = reinterpret_cast<uint16_t*>(ws);
    p.ws_ml = reinterpret_cast<float2*>(reinterpret_cast<char*>(ws) +
                                        al((size_t)p.n_query * pl.n_slots * kHeads * kDim * 2));
  }
}

static cudaError_t launch_tiles(cudaStream_t st, int kv_fmt, const AttendParams& p, int* n_launch, int persist_ctas = 0) {
  if (kv_fmt == 0 && persist_ctas > 0 && p.direct == 1 && p.n_split == 1 && p.tile_base == 0 &&
      p.tile_count == p.n_tiles) {
    cudaError_t e = cudaFuncSetAttribute(attend_persist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kAttSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)min(p.n_query, persist_ctas));
    e = launch_ex(attend_persist_kernel, grid, dim3(kAttThreads), kAttSmemBytes, st, p.pdl != 0, p.priority, p);
    if (e != cudaSuccess) return e;
    *n_launch += 1;
    return cudaGetLastError();
  }
  const dim3 grid((unsigned)(p.n_query * p.n_split));
  cudaError_t e;
#define CSA2_ATT(F)                                                                                          \
  do {                                                                                                       \
    e = cudaFuncSetAttribute(attend_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttSmemBytes); \
    if (e == cudaSuccess)                                                                                    \
      e = launch_ex(attend_kernel<F>, grid, dim3(kAttThreads), kAttSmemBytes, st, p.pdl != 0, p.priority, p);  \
  } while (0)
  if (kv_fmt == 0) CSA2_ATT(0);
  else if (kv_fmt == 1) CSA2_ATT(1);
  else CSA2_ATT(2);
#undef CSA2_ATT
  if (e != cudaSuccess) return e;
  *n_launch += 1;
  return cudaGetLastError();
}

cudaError_t launch_attend_main(cudaStream_t st, int kv_fmt, AttendParams p, const AttendPlan& pl, void* ws,
                               int* n_launch) {
  if (p.n_query == 0) return cudaSuccess;
  attach_ws(p, pl, ws);
  p.n_tiles = pl.n_tiles;
  p.tile_base = 0;
  p.tile_count = pl.n_tiles;
  p.n_split = pl.ns;
  p.tiles_per_split = pl.tps;
  p.lead_tiles = pl.lead;
  p.slot_base = 0;
  p.direct = pl.ns == 1 ? 1 : 0;
  return launch_tiles(st, kv_fmt, p, n_launch, pl.ns == 1 ? pl.ctas : 0);
}

cudaError_t launch_attend_merge(cudaStream_t st, AttendParams p, const AttendPlan& pl, void* ws, int* n_launch) {
  if (p.n_query == 0 || pl.n_slots == 0) return cudaSuccess;
  attach_ws(p, pl, ws);
  const cudaError_t e = launch_ex(attend_merge_kernel, dim3(p.n_query * (kHeads / kMergeHeadsPerCta)), dim3(256), 0,
                                  st, p.pdl != 0, 0, p);
  if (e != cudaSuccess) return e;
  *n_launch += 1;
  return cudaGetLastError();
}

cudaError_t launch_attend_partial(cudaStream_t st, int kv_fmt, AttendParams p, int with_window, int* n_launch) {
  if (p.n_query == 0) return cudaSuccess;
  p.n_tiles = attend_num_tiles(p.topk, p.topk_idx != nullptr);
  p.tile_base = with_window ? 0 : 1;
  p.tile_count = p.n_tiles - p.tile_base;
  p.n_split = 1;
  p.tiles_per_split = p.tile_count;
  p.lead_tiles = p.tile_count;
  p.slot_base = 0;
  p.n_slots = 0;
  p.direct = 2;
  return launch_tiles(st, kv_fmt, p, n_launch);
}

cudaError_t launch_attend(cudaStream_t st, int num_sms, int kv_fmt, AttendParams p, void* ws, int* n_launch,
                          bool own_window) {
  const AttendPlan pl = attend_plan(p.n_query, p.topk, p.topk_idx != nullptr, num_sms, own_window);
  cudaError_t e = launch_attend_main(st, kv_fmt, p, pl, ws, n_launch);
  if (e == cudaSuccess) e = launch_attend_merge(st, p, pl, ws, n_launch);
  return e;
}

}  // namespace csa2
