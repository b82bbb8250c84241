// kernels_inst.cuh -- instantiates the fused kernel for one (cta_group, BN)
// with the interpreter and with every catalog entry.
#pragma once

#include <utility>

#include "catalog.cuh"
#include "gemm_kernel.cuh"
#include "launch.h"

namespace ge {

template <int CG, int BN, int MC, size_t... K>
const void *pick_gemm_kernel(int epi, std::index_sequence<K...>) {
  static const void *const table[] = {
      reinterpret_cast<const void *>(&gemm_epi_kernel<CG, BN, MC, EpiStatic<catalog::Prog<K>>>)...};
  if (epi < 0) return reinterpret_cast<const void *>(&gemm_epi_kernel<CG, BN, MC, EpiInterp>);
  return epi < static_cast<int>(sizeof...(K)) ? table[epi] : nullptr;
}

}  // namespace ge

#define GE_INSTANTIATE_GEMM(CG, BN, MC, NAME)                                              \
  namespace ge {                                                                           \
  const void *NAME(int epi) {                                                              \
    return pick_gemm_kernel<CG, BN, MC>(epi, std::make_index_sequence<catalog::kCount>{}); \
  }                                                                                        \
  }
