// bfp8_sched.h -- the persistent GEMM's work decomposition, shared by the host
// planner and the device kernel (plain integer arithmetic, no CUDA types).
//
// The output is cut into tiles of 128 "P" rows (the MMA M slot, TMEM lanes)
// by BN "Q" rows (the MMA N slot, TMEM columns).  A tile's K extent is G
// blocks of 128 (one block = one set of fp32 scales, so one promotion).  A
// unit of work is one (tile, k-block) pair.
//
// Default: CTAs are persistent (grid <= SM count).  Tiles [0, dp_tiles) are handed out
// whole, round-robin (CTA p takes tiles p, p+grid, ...): neighbouring CTAs
// work on neighbouring tiles at the same time, which keeps shared operand
// rows in L2.  The remaining tiles' units are split evenly and contiguously
// across all CTAs (stream-K); a tile whose units belong to several CTAs is
// finished by the last of them to arrive, which adds the others' fp32
// partial sums in ascending K order, so the result does not depend on which
// CTA arrives last.
//
// Cluster split-K (for problems with fewer tiles than SMs): each tile is
// given to a thread-block cluster of cs CTAs, rank r taking a contiguous
// slice of the k-blocks; see make_sched_cluster.
//
// All counts fit in 32 bits (the planner rejects larger problems); the device
// walks its units with an incremental cursor, so the steady state performs no
// integer division at all.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define BFP8_HD __host__ __device__ __forceinline__
#else
#define BFP8_HD inline
#endif

namespace bfp8 {

struct Sched {
  uint32_t p_tiles;   // tiles along P (128 rows each)
  uint32_t q_tiles;   // tiles along Q (BN rows each)
  uint32_t tiles;     // p_tiles * q_tiles
  uint32_t G;         // k-blocks per tile
  uint32_t grid;      // persistent CTAs
  uint32_t dp_tiles;  // whole tiles handed out round-robin (CTA p takes tiles
                      // p, p + grid, ... below dp_tiles); a multiple of grid
                      // when stream-K units follow
  uint32_t sk_units;  // (tiles - dp_tiles) * G
  uint32_t sk_q;      // stream-K units per CTA ...
  uint32_t sk_r;      // ... plus one for CTAs p < sk_r
  uint32_t cluster;   // > 1: cluster split-K; CTA p works on tile p / cluster,
                      // k-blocks of slice p % cluster; partials are summed in
                      // distributed shared memory (no stream-K, no workspace)
};

// k-blocks [begin, end) of slice `rank` when G blocks are split `cs` ways
// (balanced: every slice has floor or ceil of G / cs blocks, so none is empty
// when cs <= G).
BFP8_HD uint32_t cluster_kb_begin(uint32_t G, uint32_t cs, uint32_t rank) {
  return static_cast<uint32_t>((static_cast<uint64_t>(rank) * G) / cs);
}
BFP8_HD uint32_t cluster_kb_end(uint32_t G, uint32_t cs, uint32_t rank) {
  return cluster_kb_begin(G, cs, rank + 1);
}

BFP8_HD uint32_t sk_begin(const Sched& s, uint32_t p) {
  return p * s.sk_q + (p < s.sk_r ? p : s.sk_r);
}

// CTA that owns stream-K unit u.
BFP8_HD uint32_t sk_owner(const Sched& s, uint32_t u) {
  const uint32_t big = s.sk_r * (s.sk_q + 1);
  return u < big ? u / (s.sk_q + 1) : s.sk_r + (u - big) / s.sk_q;
}

// Whole tiles of CTA p (all CTAs get the same number unless the schedule is
// whole tiles only with a partly filled last wave).
BFP8_HD uint32_t dp_tiles_of(const Sched& s, uint32_t p) {
  return p < s.dp_tiles ? (s.dp_tiles - p + s.grid - 1) / s.grid : 0u;
}
BFP8_HD uint32_t dp_units(const Sched& s, uint32_t p) { return dp_tiles_of(s, p) * s.G; }

BFP8_HD uint32_t num_units(const Sched& s, uint32_t p) {
  if (s.cluster > 1)
    return cluster_kb_end(s.G, s.cluster, p % s.cluster) - cluster_kb_begin(s.G, s.cluster, p % s.cluster);
  return dp_units(s, p) + sk_begin(s, p + 1) - sk_begin(s, p);
}

// CTAs that contribute to stream-K tile ts, in ascending K order.
BFP8_HD uint32_t sk_first_cta(const Sched& s, uint32_t ts) { return sk_owner(s, ts * s.G); }
BFP8_HD uint32_t sk_last_cta(const Sched& s, uint32_t ts) {
  return sk_owner(s, ts * s.G + s.G - 1);
}

// Which of CTA p's two partial slots holds its contribution to tile ts: slot 0
// for the segment its stream-K range starts in, slot 1 for the one it ends in.
BFP8_HD uint32_t sk_slot(const Sched& s, uint32_t p, uint32_t ts) {
  return (sk_begin(s, p) / s.G == ts) ? 0u : 1u;
}

// Sequential walk over one CTA's units, in the order every role processes
// them.  Divisions happen only when a new tile starts.
struct Cursor {
  uint32_t G, grid, p_tiles, dp_tiles, dp_per_cta, sk_beg;
  uint32_t n;        // units of this CTA
  uint32_t j;        // current unit index
  uint32_t tile, kb, p_tile, q_tile;
  uint32_t dp_t;     // whole tiles finished
  uint32_t u;        // current stream-K unit (when in_sk)
  bool in_sk;
  bool clustered;    // cluster split-K: one partial tile, kb from kb0
  uint32_t kb0;

  BFP8_HD void set_pq() {
    q_tile = tile / p_tiles;
    p_tile = tile - q_tile * p_tiles;
  }
  BFP8_HD void enter_sk() {
    in_sk = true;
    u = sk_beg;
    const uint32_t ts = u / G;
    tile = dp_tiles + ts;
    kb = u - ts * G;
    set_pq();
  }
  BFP8_HD void init(const Sched& s, uint32_t cta) {
    G = s.G;
    grid = s.grid;
    p_tiles = s.p_tiles;
    dp_tiles = s.dp_tiles;
    dp_per_cta = dp_tiles_of(s, cta);
    sk_beg = sk_begin(s, cta);
    n = dp_per_cta * s.G + sk_begin(s, cta + 1) - sk_beg;
    j = 0;
    dp_t = 0;
    u = 0;
    in_sk = false;
    clustered = s.cluster > 1;
    kb0 = 0;
    if (clustered) {
      const uint32_t rank = cta % s.cluster;
      kb0 = cluster_kb_begin(G, s.cluster, rank);
      n = cluster_kb_end(G, s.cluster, rank) - kb0;
      tile = cta / s.cluster;
      kb = kb0;
      set_pq();
      return;
    }
    if (n == 0) { tile = kb = p_tile = q_tile = 0; return; }
    if (dp_per_cta > 0) {
      tile = cta;
      kb = 0;
      set_pq();
    } else {
      enter_sk();
    }
  }
  BFP8_HD void next() {
    if (++j >= n) return;
    if (clustered) {
      ++kb;
      return;
    }
    if (!in_sk) {
      if (++kb == G) {
        kb = 0;
        if (++dp_t < dp_per_cta) {
          tile += grid;
          set_pq();
        } else {
          enter_sk();
        }
      }
    } else {
      ++u;
      if (++kb == G) {
        kb = 0;
        ++tile;
        if (++p_tile == p_tiles) { p_tile = 0; ++q_tile; }
      }
    }
  }
  BFP8_HD bool valid() const { return j < n; }
  BFP8_HD bool first() const { return kb == kb0 || (in_sk && u == sk_beg); }
  BFP8_HD bool last() const { return kb + 1 == G || j + 1 == n; }
  BFP8_HD int32_t sk_tile() const { return in_sk ? static_cast<int32_t>(tile - dp_tiles) : -1; }
};

// Builds the decomposition for p_tiles x q_tiles tiles of G k-blocks on at
// most `max_ctas` CTAs.  The caller checks that tiles * G fits in 31 bits.
inline Sched make_sched(uint32_t p_tiles, uint32_t q_tiles, uint32_t G, uint32_t max_ctas) {
  Sched s{};
  s.p_tiles = p_tiles;
  s.q_tiles = q_tiles;
  s.tiles = p_tiles * q_tiles;
  s.G = G;
  const uint64_t units = static_cast<uint64_t>(s.tiles) * G;
  uint64_t grid = max_ctas;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  s.grid = static_cast<uint32_t>(grid);
  // Whole waves of tiles are handed out data-parallel; only the remainder
  // (less than one wave) is split stream-K.
  s.dp_tiles = (s.tiles / s.grid) * s.grid;
  s.sk_units = (s.tiles - s.dp_tiles) * G;
  s.sk_q = s.sk_units / s.grid;
  s.sk_r = s.sk_units % s.grid;
  s.cluster = 0;
  return s;
}

// Whole tiles only, balanced: waves = ceil(tiles / max_ctas) and grid =
// ceil(tiles / waves), so every CTA takes waves or waves - 1 tiles and no
// tile is split (some SMs may stay idle; no partial sums are exchanged).
inline Sched make_sched_whole_tiles(uint32_t p_tiles, uint32_t q_tiles, uint32_t G,
                                    uint32_t max_ctas) {
  Sched s{};
  s.p_tiles = p_tiles;
  s.q_tiles = q_tiles;
  s.tiles = p_tiles * q_tiles;
  s.G = G;
  const uint32_t mc = max_ctas < 1 ? 1 : max_ctas;
  const uint32_t waves = (s.tiles + mc - 1) / mc;
  s.grid = (s.tiles + waves - 1) / waves;
  s.dp_tiles = s.tiles;
  s.sk_units = 0;
  s.sk_q = 0;
  s.sk_r = 0;
  s.cluster = 0;
  return s;
}

// Cluster split-K: tiles x cs CTAs (2 <= cs <= min(8, G)); the cs CTAs of a
// thread-block cluster share one tile, each summing a contiguous slice of its
// k-blocks, and add their partial tiles through distributed shared memory.
inline Sched make_sched_cluster(uint32_t p_tiles, uint32_t q_tiles, uint32_t G, uint32_t cs) {
  Sched s{};
  s.p_tiles = p_tiles;
  s.q_tiles = q_tiles;
  s.tiles = p_tiles * q_tiles;
  s.G = G;
  s.grid = s.tiles * cs;
  s.dp_tiles = 0;
  s.sk_units = 0;
  s.sk_q = 0;
  s.sk_r = 0;
  s.cluster = cs;
  return s;
}

}  // namespace bfp8
