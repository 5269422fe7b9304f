// zq4_rope.cuh -- the RoPE rotation of one pair (a, b) = (row i, row i + D/2)
// of a head at position pos ("Zero TVM Documentation", card 3 "QKV + RoPE +
// KV-append (fused, decode)"): angle pos * f_i, f_i = base^(-2i/D) given in
// fp64; the fp64 angle is reduced modulo 2 pi (Cody-Waite: 2 pi split into a
// double and its remainder), and the reduced angle, in [-pi, pi], goes to
// fp32 sincosf (~1e-7 rad, far inside the bound the rotation carries).
#pragma once

namespace zq4 {

__device__ __forceinline__ void rope_rotate(int pos, double inv_freq, float a, float b, float *oa, float *ob)
{
    const double kTwoPiHi = 6.283185307179586, kTwoPiLo = 2.4492935982947064e-16;
    const double th = double(pos) * inv_freq;
    const double k = rint(th * (1.0 / kTwoPiHi));
    const float r = float(fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, th)));
    float sn, cs;
    sincosf(r, &sn, &cs);
    *oa = a * cs - b * sn;
    *ob = a * sn + b * cs;
}

}  // namespace zq4
