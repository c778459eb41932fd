// The accept rule of stochastic verification, shared by the kernels that
// take it ("Speculative Decoding and MTP: Why Guessing Is Free", section
// "It's exact, not approximate": position j is accepted with probability
// min(1, p(d_j) / q(d_j)), i.e. when u_j q(d_j) < p(d_j), and the first
// rejection ends the accepted run).
#pragma once

#include "common.cuh"

namespace mtp {

// The accept decisions of positions 0..n-1 (n <= 32) taken at once, lane j of
// the calling warp holding position j: `valid` its draft token in [0, V),
// `finite` its two rows' maxima finite, `accept` u q(d) < p(d).  Returns the
// first position rejected (-1: every draft accepted) and, in `flags`, the
// status bits that taking the positions in order raises on the way there: an
// out-of-range token at the position rejected, non-finite rows at the
// positions examined.  Warp-collective.
__device__ __forceinline__ int first_rejection(int n, bool valid, bool finite, bool accept, int &flags) {
  const int lane = threadIdx.x & 31;
  const bool in = lane < n;
  const unsigned bad = __ballot_sync(0xffffffffu, in && !valid);
  const unsigned fail = bad | __ballot_sync(0xffffffffu, in && valid && !accept);
  const int rj = fail ? __ffs(fail) - 1 : -1;
  const bool bad_rj = rj >= 0 && ((bad >> rj) & 1u);
  unsigned seen = rj < 0 ? 0xffffffffu : (2u << rj) - 1u;
  if (bad_rj) seen &= ~(1u << rj);
  const unsigned nf = __ballot_sync(0xffffffffu, in && valid && !finite) & seen;
  flags = (nf ? kStatusNonFinite : 0) | (bad_rj ? kStatusBadToken : 0);
  return rj;
}

}  // namespace mtp
