// sched_device.cuh -- the work order of a persistent GEMM CTA (or CTA pair) over the output
// tiles and their 128-K slices: whole tiles in a data-parallel order, or the stream-K split
// of the slices over the units.  Shared by the software-promotion and the microscaling GEMM.
#pragma once
#include <cstdint>

namespace mpq {

// Work order of one CTA (pair): whole tiles unit, unit + nunits, ... (data-parallel), or,
// for stream-K, the contiguous run [unit U / nunits, (unit + 1) U / nunits) of the
// U = T KB slices in tile-major order, cut into per-tile segments [kb0, kb1).  With
// T >= nunits every run spans at least one tile, so a tile is shared by at most two
// consecutive units: the later one computes its last slices first (a "tail" segment, the
// run's first) and the earlier one its first slices last (a "head" segment, the run's last).
struct Sched {
    int64_t u, u1;     // stream-K position and end of the run
    int t, T, KB, nunits;
    bool sk;
};

__device__ __forceinline__ Sched sched_init(bool sk, int unit, int nunits, int T, int KB)
{
    Sched s;
    const int64_t U = static_cast<int64_t>(T) * KB;
    s.u = sk ? unit * U / nunits : 0;
    s.u1 = sk ? (unit + 1) * U / nunits : 0;
    s.t = unit;
    s.T = T;
    s.KB = KB;
    s.nunits = nunits;
    s.sk = sk;
    return s;
}

__device__ __forceinline__ bool sched_next(Sched &s, int &t, int &kb0, int &kb1)
{
    if (s.sk) {
        if (s.u >= s.u1)
            return false;
        t = static_cast<int>(s.u / s.KB);
        kb0 = static_cast<int>(s.u - static_cast<int64_t>(t) * s.KB);
        const int64_t left = s.u1 - s.u;
        kb1 = left < s.KB - kb0 ? kb0 + static_cast<int>(left) : s.KB;
        s.u += kb1 - kb0;
        return true;
    }
    if (s.t >= s.T)
        return false;
    t = s.t;
    kb0 = 0;
    kb1 = s.KB;
    s.t += s.nunits;
    return true;
}

} // namespace mpq
