// Host program for the oracle's format pins: encodes fp32 values with the
// conversion functions that CUDA's cuda_fp8.h / cuda_fp4.h declare for host
// and device (E4M3 with saturation to the largest finite value, E2M1 with
// round-to-nearest-even), so that the tests can compare them with the
// oracle's own encoders.  Test infrastructure only.
//
// stdin : one fp32 bit pattern per line, as 8 hex digits
// stdout: per input, "<e4m3 byte> <e2m1 code>" as two hex numbers
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <cstdio>
#include <cstring>

int main() {
  unsigned int bits = 0;
  while (std::scanf("%x", &bits) == 1) {
    float x;
    std::memcpy(&x, &bits, sizeof(x));
    const unsigned int e4m3 = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    const unsigned int e2m1 = __nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest);
    std::printf("%02x %x\n", e4m3 & 0xFFu, e2m1 & 0xFu);
  }
  return 0;
}
