// kernels_inst.cuh -- instantiates the fused kernel for one (cta_group, BN)
// with the interpreter and with every catalog entry.
#pragma once

#include <utility>

#include "catalog.cuh"
#include "gemm_kernel.cuh"
#include "launch.h"

namespace ge {

// epi -1 / -2: the interpreter holding 4 / 8 program registers, else catalog
// entry epi; 4 or 8 epilogue warps
template <int CG, int BN, size_t... K>
const void *pick_gemm_kernel(int epi, int warps, std::index_sequence<K...>) {
  static const void *const table4[] = {reinterpret_cast<const void *>(
      &gemm_epi_kernel<CG, BN, EpiStatic<catalog::Prog<K>, 4>>)...};
  static const void *const table8[] = {reinterpret_cast<const void *>(
      &gemm_epi_kernel<CG, BN, EpiStatic<catalog::Prog<K>, 8>>)...};
  if (epi == -1)
    return warps == 4   ? reinterpret_cast<const void *>(&gemm_epi_kernel<CG, BN, EpiInterpW<4, 4>>)
           : warps == 8 ? reinterpret_cast<const void *>(&gemm_epi_kernel<CG, BN, EpiInterpW<8, 4>>)
                        : nullptr;
  if (epi == -2)
    return warps == 4 ? reinterpret_cast<const void *>(&gemm_epi_kernel<CG, BN, EpiInterpW<4, 8>>)
                      : nullptr;
  if (epi < 0) return nullptr;
  if (epi >= static_cast<int>(sizeof...(K))) return nullptr;
  return warps == 4 ? table4[epi] : warps == 8 ? table8[epi] : nullptr;
}

}  // namespace ge

#define GE_INSTANTIATE_GEMM(CG, BN, NAME)                                                  \
  namespace ge {                                                                           \
  const void *NAME(int epi, int warps) {                                                   \
    return pick_gemm_kernel<CG, BN>(epi, warps,                                           \
                                        std::make_index_sequence<catalog::kCount>{});     \
  }                                                                                        \
  }
