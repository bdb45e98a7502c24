// The sequence of (channel group, time tile) work one CTA of a prefill kernel walks.
//
// Balanced persistent schedule: the groups' tiles, laid end to end (group-major), are cut into equal
// contiguous ranges, one per resident CTA.  A range starts inside some group g0 and ends inside
// some group g1 >= g0.  The CTA first runs the head of g1 (tiles [0, tb)) from the initial state and
// publishes the state at its end; then every complete group in between; last, the tail of g0
// (tiles [ta, Lt)), whose carried-in state the previous CTA published when it ran that head first.
// When every range is at least one group long the predecessor's head is never longer than what
// the CTA runs before its own tail, so the wait is short.
//
// Grid schedule: one CTA per (group, time chunk); a chunk that does not cover the whole sequence is
// walked as a "tail" that starts from a carried-in state.
#pragma once

#include <cstdint>

namespace ssm {

struct Walk {
  int64_t g_head;   // partial head group (tiles [0, tb)), -1 if none
  int64_t tb;
  int64_t gf0, gf1; // complete groups [gf0, gf1)
  int64_t g_tail;   // tail group (tiles [ta, ta + n_tail)), -1 if none
  int64_t ta;
  int64_t n_head, n_full, n_tail;   // tile counts of the three parts
  int64_t Lt;       // tiles per group
  __device__ int64_t total() const { return n_head + n_full + n_tail; }
  // tile k of the walk -> (group, tile within group)
  __device__ void at(int64_t k, int64_t& g, int64_t& t) const {
    if (k < n_head) { g = g_head; t = k; return; }
    k -= n_head;
    if (k < n_full) { g = gf0 + k / Lt; t = k % Lt; return; }
    k -= n_full;
    g = g_tail; t = ta + k;
  }
  __device__ bool is_tail_start(int64_t k) const { return n_tail > 0 && k == n_head + n_full; }
  // (g, t) of tile k -> (g, t) of tile k + 1, without dividing
  __device__ void advance(int64_t k, int64_t& g, int64_t& t) const {
    const int64_t k1 = k + 1;
    if (k1 == n_head) {
      if (n_full > 0) { g = gf0; t = 0; }
      else { g = g_tail; t = ta; }
      return;
    }
    if (k1 == n_head + n_full && n_tail > 0) { g = g_tail; t = ta; return; }
    if (++t == Lt) { ++g; t = 0; }   // inside a part: the next tile, or the next complete group
  }
};

// Range `cta` of `R` tiles out of `total_tiles` (group-major, `Lt` tiles per group).
__device__ inline Walk make_walk_balanced(int64_t cta, int64_t R, int64_t total_tiles, int64_t Lt) {
  Walk w;
  w.Lt = Lt;
  const int64_t A = cta * R;
  const int64_t Bn = A + R < total_tiles ? A + R : total_tiles;
  w.g_head = -1; w.g_tail = -1; w.tb = 0; w.ta = 0; w.n_head = 0; w.n_tail = 0;
  w.gf0 = w.gf1 = 0; w.n_full = 0;
  if (Bn <= A) return w;
  const int64_t g0 = A / Lt, ta = A % Lt;
  const int64_t g1 = (Bn - 1) / Lt, tb = (Bn - 1) % Lt + 1;
  int64_t f0 = g0, f1 = g1 + 1;   // candidate complete groups
  if (ta > 0) {                   // g0 starts mid-group: it is the tail (needs the carry)
    w.g_tail = g0; w.ta = ta; w.n_tail = Lt - ta; f0 = g0 + 1;
    if (g1 == g0) { f1 = f0; }    // a single tail segment (it runs to the group end)
  }
  if (tb < Lt && !(g1 == g0 && ta > 0)) {   // g1 ends mid-group: its head is run first
    w.g_head = g1; w.tb = tb; w.n_head = tb; f1 = g1;
  }
  if (f1 < f0) f1 = f0;
  w.gf0 = f0; w.gf1 = f1; w.n_full = (f1 - f0) * Lt;
  return w;
}

// Group `g`, chunk `chunk` of `chunk_tiles` tiles.
__device__ inline Walk make_walk_grid(int64_t g, int64_t chunk, int64_t chunk_tiles, int64_t Lt) {
  Walk w;
  const int64_t t0 = chunk * chunk_tiles;
  const int64_t t1 = t0 + chunk_tiles < Lt ? t0 + chunk_tiles : Lt;
  w.Lt = Lt; w.g_head = -1; w.tb = 0; w.n_head = 0; w.g_tail = -1; w.ta = 0; w.n_tail = 0;
  if (t0 == 0 && t1 == Lt) { w.gf0 = g; w.gf1 = g + 1; w.n_full = Lt; }
  else { w.gf0 = w.gf1 = 0; w.n_full = 0; w.g_tail = g; w.ta = t0; w.n_tail = t1 - t0; }
  return w;
}

}  // namespace ssm
