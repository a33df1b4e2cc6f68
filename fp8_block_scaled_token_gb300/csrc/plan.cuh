// plan.cuh -- the K-split ("stream-K") schedule shared by host and device.
//
// "A 23% faster GPU kernel, and a model that did not move", "Why this shape
// is hard": at about 8 rows the work is too narrow to fill the SMs, so the
// long (K) dimension is split across all of them and reduced
// deterministically.
//
// Work unit = (weight tile of 128 rows, one K block).  Units are numbered
// tile-major: u = tile * kg + kb.  CTA c owns the contiguous range
// [begin(c), begin(c+1)) with begin(c) = floor(U * c / P), so every CTA gets
// floor(U/P) or ceil(U/P) units.  A tile whose units fall in one CTA's range
// is finished by that CTA; otherwise each contributing CTA stores its fp32
// partial in a slot and the last one to arrive sums the slots in contributor
// order (a fixed order, independent of timing).  Everything is a pure
// function of (N, K, P), so results repeat bit for bit on a device.
#pragma once

#ifndef __CUDACC__
#define FP8BS_HD inline
#else
#define FP8BS_HD __host__ __device__ __forceinline__
#endif

namespace fp8bs {

FP8BS_HD long long plan_begin(long long units, int ctas, int c)
{
    return units * c / ctas;
}

// The CTA whose range holds unit u: the largest c with begin(c) <= u.
FP8BS_HD int plan_owner(long long units, int ctas, long long u)
{
    return static_cast<int>(((u + 1) * ctas + units - 1) / units - 1);
}

// A CTA contributes a partial to at most two tiles: the one its range starts
// in and the one it ends in.  Slot 2c holds the first, 2c+1 the second (a CTA
// whose range lies inside one tile uses 2c).  So the contributors c_first <
// c <= c_last of a tile use slot 2c, and c_first uses 2c_first + 1 unless its
// range begins exactly at the tile's first unit.

FP8BS_HD int plan_ctas(long long units, int sms)
{
    return units < sms ? static_cast<int>(units) : sms;
}

} // namespace fp8bs
