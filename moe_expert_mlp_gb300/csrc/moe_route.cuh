// Device functions of the routing permutation, shared by the standalone
// routing kernels (moe_route.cu) and the fused router, which runs them after
// its logits GEMM inside the same launch (moe_gemm.cu).
//
// "Improving MoE training throughput with advanced fused kernels",
// "Overcoming training bottlenecks in the MoE block" (tokens per expert are
// computed at run time) and "Eliminating host-device synchronisation and CPU
// launch overhead" (group sizes stay in GPU memory); "Accelerating dropless
// MoE training with JAX and NVIDIA Transformer Engine", "Claims and
// evidence" (expert-contiguous ragged groups).
//
// First reads of data other CTAs of the same launch may have written
// (histogram, top-k choices, row sources) go through L2 (ld.global.cg), so
// that no line this CTA never loaded can be served stale from its L1.
#pragma once

#include <stdint.h>

#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

// Serial scans of at most 256 experts by one thread: offsets, padded
// offsets (groups start at multiples of kAlign) and the tile prefix.
__device__ inline void scan_experts(const int32_t* cnt, int E, int capacity, int32_t* offsets,
                                    int32_t* padded_offsets, int32_t* tile_prefix, int* status) {
  int o = 0, p = 0, tp = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = o;
    padded_offsets[e] = p;
    tile_prefix[e] = tp;
    const int c = cnt[e];
    if (c < 0) set_status(status, MOE_DEV_BAD_OFFSETS);
    o += c;
    p += (c + kAlign - 1) / kAlign * kAlign;
    tp += (c + kAlign - 1) / kAlign;
  }
  offsets[E] = o;
  padded_offsets[E] = p;
  tile_prefix[E] = tp;
  if (p > capacity) set_status(status, MOE_DEV_BAD_OFFSETS);
}

// Shared scratch of one chunk's assignment (kTokensPerChunk / 32 warps).
struct AssignSmem {
  uint32_t bal[kTokensPerChunk / 32][kMaxExperts];   // per warp: lanes choosing e
  int32_t wcnt[kTokensPerChunk / 32][kMaxExperts];
  int32_t base[kMaxExperts];
  int32_t tot[kMaxExperts];
  int32_t pad[kMaxExperts];
};

// Group offsets and the stable assignment of chunk `chunk`'s (token, slot)
// pairs to rows, by kTokensPerChunk threads (tid = token inside the chunk;
// `sync` is a barrier over exactly those threads).  The per-chunk expert
// histogram [nchunks][E] is reduced first: the expert totals give the padded
// group offsets, the chunks before this one its base; chunk 0 also writes
// counts, offsets, padded offsets and the tile prefix.  The row of (token
// t, expert e) is padded_offsets[e] + (tokens of earlier chunks choosing e)
// + (earlier tokens of this chunk choosing e), so rows inside a group ascend
// by token.  One pass over the experts records, per warp, the ballot of its
// lanes choosing each expert; ranks inside a warp are popcounts of those
// ballots below the lane, across warps a shared prefix, and each token then
// places only its own k choices.
template <typename Sync>
__device__ inline void scan_assign_chunk(int chunk, int tid, const int32_t* __restrict__ topk_idx,
                                         int T, int E, int k,
                                         const int32_t* __restrict__ chunk_counts, int nchunks,
                                         int capacity, int32_t* __restrict__ counts,
                                         int32_t* __restrict__ offsets,
                                         int32_t* __restrict__ padded_offsets,
                                         int32_t* __restrict__ tile_prefix,
                                         int32_t* __restrict__ row_src,
                                         int32_t* __restrict__ row_of, int* status,
                                         AssignSmem& sm, Sync sync) {
  constexpr int NT = kTokensPerChunk, NW = NT / 32;
  for (int e = tid; e < E; e += NT) {
    int before = 0, total = 0;
#pragma unroll 4
    for (int c = 0; c < nchunks; ++c) {
      const int v = __ldcg(chunk_counts + static_cast<size_t>(c) * E + e);
      before += c < chunk ? v : 0;
      total += v;
    }
    sm.base[e] = before;
    sm.tot[e] = total;
  }
  sync();
  if (tid == 0) {
    int p = 0;
    for (int e = 0; e < E; ++e) {
      sm.pad[e] = p;
      p += (sm.tot[e] + kAlign - 1) / kAlign * kAlign;
    }
    if (chunk == 0) {
      for (int e = 0; e < E; ++e) counts[e] = sm.tot[e];
      scan_experts(sm.tot, E, capacity, offsets, padded_offsets, tile_prefix, status);
    }
  }
  sync();
  const int warp = tid >> 5, lane = tid & 31;
  const int t = chunk * NT + tid;
  const bool live = t < T;
  // the token's experts as a 256-bit mask in four scalars (a runtime index
  // into an array would keep it in local memory)
  static_assert(kMaxExperts == 256, "four 64-bit mask words");
  uint64_t sel0 = 0, sel1 = 0, sel2 = 0, sel3 = 0;
  if (live) {
    for (int s = 0; s < k; ++s) {
      const int e = __ldcg(topk_idx + static_cast<size_t>(t) * k + s);
      if (e < 0 || e >= E) {
        set_status(status, MOE_DEV_BAD_EXPERT);
        continue;
      }
      const uint64_t bit = 1ull << (e & 63);
      const int w = e >> 6;
      sel0 |= w == 0 ? bit : 0ull;
      sel1 |= w == 1 ? bit : 0ull;
      sel2 |= w == 2 ? bit : 0ull;
      sel3 |= w == 3 ? bit : 0ull;
    }
  }
  auto has_expert = [&](int e) {
    const int w = e >> 6;
    const uint64_t word = w == 0 ? sel0 : (w == 1 ? sel1 : (w == 2 ? sel2 : sel3));
    return ((word >> (e & 63)) & 1ull) != 0;
  };
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int e = 0; e < E; ++e) {
    const bool has = has_expert(e);
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, has);
    if (lane == 0) {
      sm.bal[warp][e] = b;
      sm.wcnt[warp][e] = __popc(b);
    }
  }
  sync();
  // exclusive prefix over warps, per expert
  for (int e = tid; e < E; e += NT) {
    int run = 0;
    for (int w = 0; w < NW; ++w) {
      const int v = sm.wcnt[w][e];
      sm.wcnt[w][e] = run;
      run += v;
    }
  }
  sync();
  if (!live) return;
  // re-reads of this token's choices: the first read above went to L2, so
  // these plain loads find the current values
  for (int s = 0; s < k; ++s) {
    const int e = topk_idx[static_cast<size_t>(t) * k + s];
    if (e < 0 || e >= E) continue;                // recorded above
    const int rank = sm.wcnt[warp][e] + __popc(sm.bal[warp][e] & lt_mask);
    const int row = sm.pad[e] + sm.base[e] + rank;
    row_src[row] = t;
    row_of[static_cast<size_t>(t) * k + s] = row;
  }
}

// x_perm[j] = x[row_src[j]] (zero on padding rows): one warp moves one row
// of vec_per_row 16-byte vectors.
__device__ inline void gather_row_warp(const uint4* __restrict__ x,
                                       const int32_t* __restrict__ row_src, int j,
                                       int vec_per_row, int T, uint4* __restrict__ x_perm,
                                       int lane) {
  const int t = __ldcg(row_src + j);
  uint4* dst = x_perm + static_cast<size_t>(j) * vec_per_row;
  if (t >= 0 && t < T) {
    const uint4* src = x + static_cast<size_t>(t) * vec_per_row;
    int c = lane;
    for (; c + 96 < vec_per_row; c += 128) {       // four loads in flight per lane
      const uint4 a = __ldg(src + c), b = __ldg(src + c + 32), d = __ldg(src + c + 64),
                  e = __ldg(src + c + 96);
      dst[c] = a;
      dst[c + 32] = b;
      dst[c + 64] = d;
      dst[c + 96] = e;
    }
    for (; c < vec_per_row; c += 32) dst[c] = __ldg(src + c);
  } else {
    for (int c = lane; c < vec_per_row; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
  }
}

}  // namespace moe
