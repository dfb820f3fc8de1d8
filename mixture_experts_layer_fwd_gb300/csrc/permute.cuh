// Row copy of the permutation, shared by the gather kernel (permute.cu) and
// the fused dispatch (dispatch.cu).
#pragma once

#include "common.cuh"

namespace moe {

DEVINL uint32_t bf16x2_to_f16x2_satfinite(uint32_t v) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(v & 0xFFFF0000u)),
      "f"(__uint_as_float(v << 16)));
  return r;
}
DEVINL uint4 cvt_row_vec(uint4 v, bool to_f16) {
  if (!to_f16) return v;
  return make_uint4(bf16x2_to_f16x2_satfinite(v.x), bf16x2_to_f16x2_satfinite(v.y), bf16x2_to_f16x2_satfinite(v.z),
                    bf16x2_to_f16x2_satfinite(v.w));
}

// One warp copies token row t of x (row_bytes, a multiple of 16, in 16-byte
// vectors) and its sf_bytes scale bytes (a multiple of 4; none when x_sf is
// NULL) to row r of xp / xp_sf.  TO_F16: the row holds bf16 values, written
// as fp16 (saturating).
template <bool TO_F16>
DEVINL void copy_row(const uint8_t* __restrict__ x, int row_bytes, const uint8_t* __restrict__ x_sf, int sf_bytes,
                     int t, uint8_t* __restrict__ xp, uint8_t* __restrict__ xp_sf, int r, int lane) {
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * row_bytes);
  uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<size_t>(r) * row_bytes);
  const int nvec = row_bytes >> 4;
  // the row's scale words (up to 128 of them: 512 scale bytes) are loaded
  // first, so that their round trip overlaps the code vectors'
  const int nsw = x_sf != nullptr ? (sf_bytes >> 2) : 0;
  const uint32_t* ssrc = nsw ? reinterpret_cast<const uint32_t*>(x_sf + static_cast<size_t>(t) * sf_bytes) : nullptr;
  uint32_t sv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (lane + 32 * u < nsw) sv[u] = __ldg(ssrc + lane + 32 * u);
  // eight 16-byte loads of the lane in flight before its stores (one round
  // trip per 256 vectors = 4 KB of the row)
  for (int i0 = 0; i0 < nvec; i0 += 256) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + lane + 32 * j;
      if (i < nvec) v[j] = __ldg(src + i);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + lane + 32 * j;
      if (i < nvec) dst[i] = cvt_row_vec(v[j], TO_F16);
    }
  }
  if (nsw) {
    uint32_t* sdst = reinterpret_cast<uint32_t*>(xp_sf + static_cast<size_t>(r) * sf_bytes);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (lane + 32 * u < nsw) sdst[lane + 32 * u] = sv[u];
    for (int j = lane + 128; j < nsw; j += 32) sdst[j] = __ldg(ssrc + j);
  }
}

}  // namespace moe
