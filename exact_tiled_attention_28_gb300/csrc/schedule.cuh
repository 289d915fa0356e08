// Static order in which persistent CTAs take work items.
#pragma once

namespace fa {

// Item handled by CTA c (of G) in round rnd. Items are numbered longest first.
// Non-causal items all cost the same, and CTA c takes c, c + G, c + 2G, ...
// Causal items shrink along the list, so rounds alternate direction: CTA c
// takes item rnd*G + c in even rounds and rnd*G + (G-1-c) in odd ones. A CTA that
// got a long item in one round gets a short one in the next, and the largest
// per-CTA total comes within about 2% of the average (plain striding: 7-14%
// above it for the configurations measured). Every warp role of a CTA walks
// the same sequence.
__device__ __forceinline__ int sched_item(int rnd, int c, int G, bool causal) {
  return rnd * G + ((causal && (rnd & 1)) ? G - 1 - c : c);
}

}  // namespace fa
