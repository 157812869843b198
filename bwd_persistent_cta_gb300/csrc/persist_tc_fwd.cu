// persist_tc_fwd.cu - the instances of the forward persistent
// tensor-core kernel (persist_tc_kernels.cuh), in a translation unit of their own.
#include "persist_tc_kernels.cuh"

namespace rnn {

namespace {

template <int KS, bool EXT>
const void* by_pp(int pp) {
  switch (pp) {
    case 1: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<1, KS, EXT>);
    case 2: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<2, KS, EXT>);
    case 4: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<4, KS, EXT>);
    default: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<8, KS, EXT>);
  }
}

template <bool EXT>
const void* by_ks(int pp, int ks) {
  switch (ks) {
    case 1: return by_pp<1, EXT>(pp);
    case 2: return by_pp<2, EXT>(pp);
    case 4: return by_pp<4, EXT>(pp);
    case 8: return by_pp<8, EXT>(pp);
    default: return by_pp<16, EXT>(pp);
  }
}

}  // namespace

const void* persist_tc_fwd_kernel_ptr(int pp, int ks, int ext) {
  return ext ? by_ks<true>(pp, ks) : by_ks<false>(pp, ks);
}

#ifdef RNN_STEP_TRACE
// this translation unit's copy of the step-trace buffer (forward: kind 0)
extern "C" int rnn_debug_read_step_trace_fwd(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, g_step_trace, bytes) == cudaSuccess ? 0 : 3;
}
#endif

}  // namespace rnn
