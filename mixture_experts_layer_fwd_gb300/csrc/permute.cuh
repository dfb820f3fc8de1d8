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
  int i = lane;
  for (; i + 96 < nvec; i += 128) {
    const uint4 a = __ldg(src + i), b = __ldg(src + i + 32), c = __ldg(src + i + 64), d = __ldg(src + i + 96);
    dst[i] = cvt_row_vec(a, TO_F16);
    dst[i + 32] = cvt_row_vec(b, TO_F16);
    dst[i + 64] = cvt_row_vec(c, TO_F16);
    dst[i + 96] = cvt_row_vec(d, TO_F16);
  }
  for (; i < nvec; i += 32) dst[i] = cvt_row_vec(__ldg(src + i), TO_F16);
  if (x_sf != nullptr) {
    const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(x_sf + static_cast<size_t>(t) * sf_bytes);
    uint32_t* sdst = reinterpret_cast<uint32_t*>(xp_sf + static_cast<size_t>(r) * sf_bytes);
    for (int j = lane; j < (sf_bytes >> 2); j += 32) sdst[j] = __ldg(ssrc + j);
  }
}

}  // namespace moe
