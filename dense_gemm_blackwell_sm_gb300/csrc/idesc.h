// idesc.h -- the 32-bit tcgen05 instruction descriptor, packed on the host in
// one place for every kernel of the library.
//
// The descriptor tells tcgen05.mma the accumulator format, the A / B element
// formats, whether A or B is stored MN-major, and the MMA shape (N / 8 and
// M / 16).  Bit positions follow the PTX ISA's table of the instruction
// descriptor for kind::f16, kind::f8f6f4 and kind::mxf8f6f4.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define DGB_HD __host__ __device__
#else
#define DGB_HD
#endif

namespace dgb {

// fields common to the three kinds
constexpr uint32_t IDESC_D_F32 = 1u << 4;      // accumulator format: fp32 (f16 and f8f6f4 kinds)
constexpr uint32_t IDESC_A_MN_MAJOR = 1u << 15;
constexpr uint32_t IDESC_B_MN_MAJOR = 1u << 16;
constexpr uint32_t IDESC_SCALE_UE8M0 = 1u << 23;  // kind::mxf8f6f4: scale factors are UE8M0
constexpr uint32_t IDESC_N_MASK = 0x3Fu << 17;

inline uint32_t idesc_shape(int M, int N) { return ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24); }

// kind::f16: A and B both fp16 (format 0) or both bf16 (format 1), fp32 accumulator
inline uint32_t idesc_f16(bool bf16, int M, int N) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return IDESC_D_F32 | (ab << 7) | (ab << 10) | idesc_shape(M, N);
}

// kind::f8f6f4: A and B both E4M3 (format 0) or both E5M2 (format 1), fp32 accumulator
inline uint32_t idesc_f8(bool e5m2, int M, int N) {
  const uint32_t f = e5m2 ? 1u : 0u;
  return IDESC_D_F32 | (f << 7) | (f << 10) | idesc_shape(M, N);
}

// kind::mxf8f6f4: E4M3 / E5M2 operands with UE8M0 block scales; the scale-byte
// selectors (B: bits 4-5, A: bits 29-30) are added per MMA by the kernel
inline uint32_t idesc_mx(bool e5m2, int M, int N) {
  const uint32_t f = e5m2 ? 1u : 0u;
  return (f << 7) | (f << 10) | IDESC_SCALE_UE8M0 | idesc_shape(M, N);
}

// the same descriptor with another N
DGB_HD inline uint32_t idesc_with_n(uint32_t idesc, int N) {
  return (idesc & ~IDESC_N_MASK) | ((uint32_t)(N >> 3) << 17);
}

}  // namespace dgb
