// bfp8_sched.h -- the persistent GEMM's work decomposition, shared by the host
// planner and the device kernel (plain integer arithmetic, no CUDA types).
//
// The output is cut into tiles of 128 "P" rows (the MMA M slot, TMEM lanes)
// by BN "Q" rows (the MMA N slot, TMEM columns).  A tile's K extent is G
// blocks of 128 (one block = one set of fp32 scales, so one promotion).  A
// unit of work is one (tile, k-block) pair.
//
// CTAs are persistent (grid <= SM count).  Tiles [0, dp_tiles) are handed out
// whole, round-robin (CTA p takes tiles p, p+grid, ...): neighbouring CTAs
// work on neighbouring tiles at the same time, which keeps shared operand
// rows in L2.  The remaining tiles' units are split evenly and contiguously
// across all CTAs (stream-K); a tile whose units belong to several CTAs is
// finished by the last of them to arrive, which adds the others' fp32
// partial sums in ascending K order, so the result does not depend on which
// CTA arrives last.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define BFP8_HD __host__ __device__ __forceinline__
#else
#define BFP8_HD inline
#endif

namespace bfp8 {

struct Sched {
  int64_t p_tiles;   // tiles along P (128 rows each)
  int64_t q_tiles;   // tiles along Q (BN rows each)
  int64_t tiles;     // p_tiles * q_tiles
  int32_t G;         // k-blocks per tile
  int32_t grid;      // persistent CTAs
  int64_t dp_tiles;  // whole tiles handed out round-robin; a multiple of grid
  int64_t sk_units;  // (tiles - dp_tiles) * G
  int64_t sk_q;      // units per CTA in the stream-K part ...
  int64_t sk_r;      // ... plus one for CTAs p < sk_r
};

struct Unit {
  int64_t tile;      // tile index; p_tile = tile % p_tiles, q_tile = tile / p_tiles
  int32_t kb;        // k-block
  int32_t first;     // first unit of a segment (accumulator starts from zero)
  int32_t last;      // last unit of a segment (the segment's result is emitted)
  int64_t sk_tile;   // index among stream-K tiles, or -1 for a whole (data-parallel) tile
};

BFP8_HD int64_t sk_begin(const Sched& s, int64_t p) {
  return p * s.sk_q + (p < s.sk_r ? p : s.sk_r);
}

// CTA that owns stream-K unit u.
BFP8_HD int64_t sk_owner(const Sched& s, int64_t u) {
  const int64_t big = s.sk_r * (s.sk_q + 1);
  return u < big ? u / (s.sk_q + 1) : s.sk_r + (u - big) / s.sk_q;
}

BFP8_HD int64_t dp_units(const Sched& s) { return (s.dp_tiles / s.grid) * s.G; }

BFP8_HD int64_t num_units(const Sched& s, int64_t p) {
  return dp_units(s) + sk_begin(s, p + 1) - sk_begin(s, p);
}

BFP8_HD Unit unit_at(const Sched& s, int64_t p, int64_t j) {
  Unit u;
  const int64_t dpu = dp_units(s);
  if (j < dpu) {
    const int64_t t = j / s.G;
    u.kb = static_cast<int32_t>(j - t * s.G);
    u.tile = p + t * s.grid;
    u.sk_tile = -1;
    u.first = u.kb == 0;
    u.last = u.kb == s.G - 1;
  } else {
    const int64_t uu = sk_begin(s, p) + (j - dpu);
    const int64_t ts = uu / s.G;
    u.kb = static_cast<int32_t>(uu - ts * s.G);
    u.tile = s.dp_tiles + ts;
    u.sk_tile = ts;
    u.first = (u.kb == 0) || (j == dpu);
    u.last = (u.kb == s.G - 1) || (j == num_units(s, p) - 1);
  }
  return u;
}

// CTAs that contribute to stream-K tile ts, in ascending K order.
BFP8_HD int64_t sk_first_cta(const Sched& s, int64_t ts) { return sk_owner(s, ts * s.G); }
BFP8_HD int64_t sk_last_cta(const Sched& s, int64_t ts) {
  return sk_owner(s, ts * s.G + s.G - 1);
}

// Which of CTA p's two partial slots holds its contribution to tile ts: slot 0
// for the segment its stream-K range starts in, slot 1 for the one it ends in.
BFP8_HD int32_t sk_slot(const Sched& s, int64_t p, int64_t ts) {
  return (sk_begin(s, p) / s.G == ts) ? 0 : 1;
}

// Builds the decomposition for `tiles` tiles of G k-blocks on at most
// `max_ctas` CTAs.
inline Sched make_sched(int64_t p_tiles, int64_t q_tiles, int32_t G, int32_t max_ctas) {
  Sched s{};
  s.p_tiles = p_tiles;
  s.q_tiles = q_tiles;
  s.tiles = p_tiles * q_tiles;
  s.G = G;
  const int64_t units = s.tiles * G;
  int64_t grid = max_ctas;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  s.grid = static_cast<int32_t>(grid);
  if (s.tiles % grid == 0) {
    s.dp_tiles = s.tiles;                        // whole waves: no stream-K
  } else {
    const int64_t waves = s.tiles / grid;
    s.dp_tiles = waves >= 2 ? (waves - 1) * grid : 0;
  }
  s.sk_units = (s.tiles - s.dp_tiles) * G;
  s.sk_q = s.sk_units / grid;
  s.sk_r = s.sk_units % grid;
  return s;
}

}  // namespace bfp8
