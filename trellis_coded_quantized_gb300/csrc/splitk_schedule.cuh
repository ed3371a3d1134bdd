// Work schedule of the tensor-core axis-0 scatter (host and device).
//
// The method's split-K structure (@mlx-bun/inference 1.0.0,
// kernels/trellis/scatter.ts, rowsPer/r0/r1 split ranges and the [M, SPLITS,
// C] float partials): split s owns input rows [s*rp, min(R, (s+1)*rp)),
// rp = ceil(R/S), and its partial P[m][s][c] is the sum over those rows.
//
// An "item" is one split and one block of 256 output columns, i = s*NB + b;
// it takes ceil(rows of s / 16) "steps" of 16 rows (one MMA K step each).
// The steps of all items, item after item, form one line of T steps, and
// CTA g of G takes the contiguous run [floor(g*T/G), floor((g+1)*T/G)), so
// every CTA decodes the same number of weights whatever the split count.
// An item cut between CTAs is finished by the split reduction: the CTA that
// holds the item's first step writes its share to the partial itself, each
// later CTA on the item (for which it is necessarily the first item of its
// run) writes its share to its own fix-up slot, and the reduction adds the
// slots to the partial in CTA order -- a fixed order, so the partials are
// deterministic.
#pragma once

#include <stdint.h>

namespace tcq {

struct SplitSchedule {
    int64_t R;      // input rows
    int64_t rp;     // rows per split
    int S;          // splits
    int NB;         // blocks of 256 output columns
    int F;          // splits with rp rows
    int nf;         // steps of such a split
    int nrem;       // steps of split F (the remainder; 0 when F == S)
    int G;          // CTAs
    int64_t T;      // steps of all items

    __host__ __device__ static SplitSchedule make(int64_t R, int S, int64_t C, int G) {
        SplitSchedule sc;
        sc.R = R;
        sc.S = S;
        sc.rp = (R + S - 1) / S;
        sc.NB = (int)(C / 256);
        sc.F = (int)(R / sc.rp);                 // <= S
        sc.nf = (int)((sc.rp + 15) / 16);
        const int64_t rem = R - (int64_t)sc.F * sc.rp;
        sc.nrem = sc.F < S ? (int)((rem + 15) / 16) : 0;
        sc.T = (int64_t)sc.NB * ((int64_t)sc.F * sc.nf + sc.nrem);
        sc.G = G;
        return sc;
    }
    __host__ __device__ int steps(int s) const { return s < F ? nf : (s == F ? nrem : 0); }
    // steps of all splits before s
    __host__ __device__ int64_t prefix(int s) const {
        return s <= F ? (int64_t)s * nf : (int64_t)F * nf + nrem;
    }
    __host__ __device__ int64_t row0(int s) const { return (int64_t)s * rp; }
    __host__ __device__ int64_t row1(int s) const {
        const int64_t e = (int64_t)s * rp + rp;
        return e < R ? e : R;
    }
    // first step of CTA g (g = G gives T)
    __host__ __device__ int64_t start(int g) const { return (int64_t)g * T / G; }
    // the CTA whose run holds step x (the last g with start(g) <= x)
    __host__ __device__ int cta_of(int64_t x) const { return (int)(((x + 1) * G - 1) / T); }
    // The same two in 32-bit arithmetic, exact when T * G < 2^32 (any
    // schedule below 26 million steps at 160 CTAs): a 64-bit division costs
    // tens of dependent instructions.
    __host__ __device__ bool small() const { return (uint64_t)T * (uint64_t)G < (1ull << 32); }
    __host__ __device__ uint32_t start32(int g) const { return (uint32_t)g * (uint32_t)T / (uint32_t)G; }
    __host__ __device__ int cta_of32(uint32_t x) const {
        return (int)(((x + 1u) * (uint32_t)G - 1u) / (uint32_t)T);
    }
    // split s, block b and step k within the item of step x; n = steps of the item
    __host__ __device__ void locate(int64_t x, int& s, int& b, int& k, int& n) const {
        const int64_t full = (int64_t)NB * F * nf;
        if (x < full) {
            const int64_t per = (int64_t)NB * nf;
            s = (int)(x / per);
            const int64_t w = x - (int64_t)s * per;
            b = (int)(w / nf);
            k = (int)(w - (int64_t)b * nf);
            n = nf;
        } else {
            const int64_t w = x - full;
            s = F;
            b = (int)(w / nrem);
            k = (int)(w - (int64_t)b * nrem);
            n = nrem;
        }
    }
};

}  // namespace tcq
