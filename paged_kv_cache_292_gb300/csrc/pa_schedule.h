// Work decomposition of one decode batch, shared by the attention kernel, the
// merge kernel and host-side tests (plain C++ when compiled without nvcc).
//
// Every sequence s contributes ceil(ctx_s / kTile) tiles of kTile tokens.  The
// tiles of all sequences, in sequence order, form one flat list of T tiles.
// That list is cut into R equal ranges: range r owns tiles
// [floor(r*T/R), floor((r+1)*T/R)).  One CTA (per KV-head group) walks one
// range, so every CTA streams the same number of K/V bytes whatever the
// context-length mix.  A sequence whose tiles all fall in one range is
// finished by that CTA; a sequence that straddles ranges leaves one partial
// result per range it touches, merged afterwards by log-sum-exp.
//
// Partial-result slot rule: in range r, the sequence holding the range's first
// tile writes slot 0; a different sequence cut at the range's end writes slot
// 1.  Every other sequence touched by the range lies wholly inside it.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define PA_HD __host__ __device__ __forceinline__
#else
#define PA_HD inline
#endif

namespace pa {

constexpr int kTile = 16;  // tokens per tile (one MMA M-extent, one pipeline stage)

PA_HD int64_t range_start(int64_t r, int64_t total_tiles, int64_t num_ranges) {
  const int64_t prod = r * total_tiles;
  // 32-bit division when the operands fit (the common case; much cheaper on the GPU).
  if (prod < (int64_t(1) << 32) && num_ranges < (int64_t(1) << 32))
    return static_cast<int64_t>(static_cast<uint32_t>(prod) / static_cast<uint32_t>(num_ranges));
  return prod / num_ranges;
}

// The range that owns tile x (0 <= x < total_tiles).  Empty ranges own nothing.
PA_HD int64_t range_of_tile(int64_t x, int64_t total_tiles, int64_t num_ranges) {
  const int64_t prod = x * num_ranges;
  int64_t r = (prod < (int64_t(1) << 32) && total_tiles < (int64_t(1) << 32))
                  ? static_cast<int64_t>(static_cast<uint32_t>(prod) / static_cast<uint32_t>(total_tiles))
                  : prod / total_tiles;
  if (r >= num_ranges) r = num_ranges - 1;
  while (r + 1 < num_ranges && range_start(r + 1, total_tiles, num_ranges) <= x) ++r;
  while (r > 0 && range_start(r, total_tiles, num_ranges) > x) --r;
  return r;
}

PA_HD int tiles_of(int ctx) { return (ctx + kTile - 1) / kTile; }

// Output destination of the segment [seg_lo, seg_hi) of a sequence whose tiles
// are [seq_lo, seq_hi), walked by the range [r_lo, r_hi).
//   -1: the whole sequence is in this range (write the final output);
//    0 / 1: partial slot.
PA_HD int segment_slot(int64_t r_lo, int64_t r_hi, int64_t seq_lo, int64_t seq_hi) {
  if (r_lo <= seq_lo && r_hi >= seq_hi) return -1;
  return (r_lo >= seq_lo) ? 0 : 1;
}

// Slot in which range r left its partial for a sequence starting at tile
// seq_lo (r must touch that sequence and be non-empty).
PA_HD int partial_slot_of_range(int64_t r, int64_t seq_lo, int64_t total_tiles,
                                int64_t num_ranges) {
  return (range_start(r, total_tiles, num_ranges) >= seq_lo) ? 0 : 1;
}

}  // namespace pa
