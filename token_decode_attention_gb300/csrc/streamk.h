// streamk.h -- partition arithmetic of the stream-K decode, shared by host
// code, both kernels and the host-side unit check (tests/streamk_check.cpp).
//
// The live KV positions of a batch are flattened unit by unit, where a unit is
// (sequence b, head group g) and holds L_b positions:
//   unit u = b * NHG + g  covers  [NHG * Pb[b] + g * L_b,  NHG * Pb[b] + (g+1) * L_b)
// with Pb[b] = sum_{b' < b} L_b' and W = NHG * Pb[B] positions in total.
// Partition c of G owns [range_begin(c), range_begin(c + 1)); the ranges tile
// [0, W) and differ in length by at most one position.  A partition's range
// crosses units; the part of unit u that partition c processes is a "piece",
// and its partial softmax state lives in workspace slot piece_slot(c, u).
// Along the flattened order both c and u are non-decreasing and at least one
// of them grows from one piece to the next, so c + u is unique per piece and
// below G + U.
#pragma once

#ifdef __CUDACC__
#define DATTN_HD __host__ __device__ __forceinline__
#else
#define DATTN_HD inline
#endif

namespace dattn {

// First flattened position of partition c (0 <= c <= G).  Requires c * W to
// fit in 64 bits (checked by the host before launch).
DATTN_HD long long range_begin(long long c, long long W, long long G) { return c * W / G; }

// The partition whose range holds flattened position x (0 <= x < W): the
// largest c with floor(c W / G) <= x, i.e. ceil((x + 1) G / W) - 1.
DATTN_HD long long range_owner(long long x, long long W, long long G) {
    const long long n = (x + 1) * G + W - 1;
    if (n < 0x100000000LL)  // a 32-bit division (W <= n)
        return static_cast<long long>(static_cast<unsigned>(n) / static_cast<unsigned>(W)) - 1;
    return n / W - 1;
}

// range_begin(c, W, G) with W = wq * G + wr (wq = W / G, wr = W % G) and
// G <= 65535: c * W / G = c * wq + (c * wr) / G exactly, and c * wr < G * G
// fits in 32 bits, so the per-partition division is a 32-bit one.
DATTN_HD long long range_begin_split(unsigned c, long long wq, unsigned wr, unsigned G) {
    return static_cast<long long>(c) * wq +
           static_cast<long long>(static_cast<unsigned>(static_cast<unsigned long long>(c) * wr) / G);
}

// Workspace slot of the piece of unit u processed by partition c.
DATTN_HD long long piece_slot(long long c, long long u) { return c + u; }

}  // namespace dattn
