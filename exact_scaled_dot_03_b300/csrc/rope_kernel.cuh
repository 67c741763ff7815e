// Rotary position embedding for the prefill ([PW] §5.3): each pair (2i, 2i+1)
// of a Q or K vector at position m is rotated by theta = m * w_i with
// w_i = base^(-2i/d), so scores depend only on the relative position.
//
// Sources: [PW] pwwt.cn news 6124947, §5.3 (RoPE rotation matrix, w_i).
//
// Work split (B300): K is read by every query tile of its group, so it is
// rotated once, here, into a workspace copy; Q is read once per CTA and is
// rotated inside the prefill kernel's load stage (see fwd_kernel.cuh), using
// the transposed copy of the (cos, sin) table built here.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace attn_dev {

constexpr int kRopeMaxPairs = 64;  // d <= 128

struct RopeArgs {
  float2* cs;                     // [T][D/2] (cos, sin) of positions pmin .. pmin + T - 1
  float2* cs_t;                   // the same values as [D/2][T]: a warp's 32 consecutive
                                  // positions of one pair are 256 contiguous bytes
  int T, pmin;
  double w[kRopeMaxPairs];        // w_i = base^(-2i/d), computed on the host in fp64
};

// (cos, sin) of every position of the table and every pair. The angle is
// formed and reduced modulo 2 pi in fp64 (positions reach 10^4-10^5 rad for
// the highest frequency), then sincosf gives the fp32 values.
template <int D>
__global__ void rope_table_kernel(const RopeArgs a) {
  constexpr int NP = D / 2;
  const long long n = (long long)a.T * NP;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / NP), i = (int)(e % NP);
    const double theta = (double)(a.pmin + t) * a.w[i];
    // theta - 2 pi k with k = nearest integer to theta / (2 pi): a multiply
    // by the reciprocal and one FMA (fp64 division is slow on this part).
    const double two_pi = 6.283185307179586476925286766559, inv_two_pi = 0.15915494309189533576888376337251;
    const double r = fma(-two_pi, rint(theta * inv_two_pi), theta);
    float s, c;
    sincosf((float)r, &s, &c);
    a.cs[e] = make_float2(c, s);
    a.cs_t[(size_t)i * a.T + t] = make_float2(c, s);
  }
}

// k_rot[b, h, j, :] = rope(k[b, h, j, :], position j), rounded to bf16 (RNE).
// One thread per 8 components (4 pairs, one 16-byte chunk).
template <int D>
__global__ void rope_k_kernel(const __nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ k_rot,
                              const float2* __restrict__ cs, long long rows, int Nk, int pmin) {
  constexpr int CH = D / 8;
  const long long n = rows * CH;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
    const long long row = e / CH;
    const int c = (int)(e % CH);
    const int pos = (int)(row % Nk);
    const uint4 w = *reinterpret_cast<const uint4*>(k + row * D + 8 * c);
    const float2* tab = cs + (size_t)(pos - pmin) * (D / 2) + 4 * c;
    uint32_t in[4] = {w.x, w.y, w.z, w.w}, out[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float x = __uint_as_float(in[p] << 16), y = __uint_as_float(in[p] & 0xffff0000u);
      const float2 t = tab[p];
      out[p] = pack_bf16x2(x * t.x - y * t.y, x * t.y + y * t.x);
    }
    *reinterpret_cast<uint4*>(k_rot + row * D + 8 * c) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

}  // namespace attn_dev
