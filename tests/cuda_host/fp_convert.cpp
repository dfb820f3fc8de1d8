// Host program for the oracle's format pins: calls the conversion functions
// that CUDA's cuda_fp8.h / cuda_fp4.h declare for host and device, so that
// the tests can compare them with the oracle's own encoders.  Test
// infrastructure only.
//
// Modes (first argument; default "fp"), one hex number per input line:
//   fp      : fp32 bit pattern -> "<e4m3 byte> <e2m1 code>": E4M3 with
//             saturation to the largest finite value, E2M1 with
//             round-to-nearest-even
//   e8m0    : fp32 bit pattern -> "<e8m0 byte>": the E8M0 scale of the value
//             rounded toward zero (the power of two at or below it)
//   e8m0dec : E8M0 byte -> "<bf16 bits>" of its value
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <cstdio>
#include <cstring>

int main(int argc, char** argv) {
  const char* mode = argc > 1 ? argv[1] : "fp";
  unsigned int bits = 0;
  while (std::scanf("%x", &bits) == 1) {
    if (std::strcmp(mode, "e8m0dec") == 0) {
      const __nv_bfloat16_raw r = __nv_cvt_e8m0_to_bf16raw(static_cast<__nv_fp8_storage_t>(bits & 0xFFu));
      std::printf("%04x\n", static_cast<unsigned int>(r.x));
      continue;
    }
    float x;
    std::memcpy(&x, &bits, sizeof(x));
    if (std::strcmp(mode, "e8m0") == 0) {
      const unsigned int c = __nv_cvt_float_to_e8m0(x, __NV_SATFINITE, cudaRoundZero);
      std::printf("%02x\n", c & 0xFFu);
    } else {
      const unsigned int e4m3 = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
      const unsigned int e2m1 = __nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest);
      std::printf("%02x %x\n", e4m3 & 0xFFu, e2m1 & 0xFu);
    }
  }
  return 0;
}
