// Shared by the two-pass kernels (columns and rows), which run a softmax's
// two passes as work items of one launch: the order in which items are dealt
// out by arrival, the arrival draw itself, the ticket-tagged words through
// which first passes hand their (max, sum) pairs to second passes, and the
// packed exponent arithmetic.
#pragma once

#include <stdint.h>

#include "device_common.cuh"

namespace rrs {

// 2^((v - m) log2 e) for a pair of floats in one f32x2 register: v - m as
// v + (-m), exact like the scalar subtraction, then the scalar's rounding of
// the product (the exponent arithmetic of the column and row kernels).
__device__ __forceinline__ uint64_t exp_shifted2(float va, float vb, uint64_t neg_m2, uint64_t log2e2) {
  float ta, tb;
  f2_unpack(f2_mul(f2_add(f2_pack(va, vb), neg_m2), log2e2), ta, tb);
  return f2_pack(exp2_sfu(ta), exp2_sfu(tb));
}

// Every wait of a two-pass kernel gives up after this long (global timer).
constexpr uint64_t kTwoPassWaitNs = 1000000000ull;

// The (pass, item) of arrival index t among the 2 Q arrivals of a launch
// with Q items per pass and lag D (1 <= D <= Q): pass 1 of items 0 .. D - 1,
// then pass 1 of item D + i and pass 2 of item i alternately, then pass 2
// of the last D items.  Pass 2 of an item thus trails its pass 1 by 2 D + 1
// arrivals; a D at least the number of items one second pass depends on
// keeps all of them ahead of it.
__host__ __device__ inline void two_pass_item(int64_t t, int64_t Q, int64_t D, int* pass, int64_t* k) {
  if (t < D) {
    *pass = 1;
    *k = t;
    return;
  }
  const int64_t u = t - D;
  if (u < 2 * (Q - D)) {
    *pass = (u & 1) ? 2 : 1;
    *k = (u & 1) ? (u >> 1) : D + (u >> 1);
    return;
  }
  *pass = 2;
  *k = (Q - D) + (u - 2 * (Q - D));
}

// (ticket << 32 | bits(v)): a 64-bit word is single-copy atomic, so a reader
// that sees this launch's ticket in a word has the value written with it.
__device__ __forceinline__ uint64_t tagged_word(uint32_t ticket, float v) {
  return ((uint64_t)ticket << 32) | (uint64_t)__float_as_uint(v);
}

// The arrival index of this CTA among the `draws` of its launch and the
// launch's ticket, from the counter word (epoch << 32 | count); the last of
// the draws opens the next epoch (count 0), so the next launch on the stream
// starts from 0 and tags with a fresh ticket.
__device__ __forceinline__ unsigned draw_arrival(unsigned long long* arrivals, unsigned draws, unsigned* ticket) {
  const unsigned long long old = atomicAdd(arrivals, 1ull);
  const unsigned a = (unsigned)(old & 0xffffffffull);
  const unsigned epoch = (unsigned)(old >> 32);
  if (a == draws - 1) {
    atomicExch(arrivals, (unsigned long long)(epoch == 0xfffffffeu ? 0u : epoch + 1u) << 32);
    __threadfence();
  }
  *ticket = epoch + 1u;   // never 0, the tag of a zero-filled slot
  return a;
}

}  // namespace rrs
