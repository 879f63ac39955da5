// gemm_tc.cuh - tensor-core (tcgen05) matrix products.  Placeholder until
// the tcgen05 path lands: the CUDA-core path runs every product.
#pragma once
#include "common.cuh"
#include "gemm.cuh"

struct TcState {
  unsigned tmem_base;
  unsigned long long iters;
};

template <class OP>
__device__ __forceinline__ void tc_setup(const KArgs& a, char* smem, TcState& tc) {
  tc.tmem_base = 0;
  tc.iters = 0;
}
template <class OP>
__device__ __forceinline__ void tc_teardown(const KArgs& a, char* smem, TcState& tc) {}

__device__ __forceinline__ void gemm_tc_job(const KArgs& a, const GemmDesc& g, Sched& s, char* smem,
                                            TcState& tc) {}

#define MT_TC_AVAILABLE 0
#define MT_TC_SMEM 0
