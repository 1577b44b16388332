// paged_prefill_varlen fast path on the 5th-generation tensor cores
// (tcgen05.mma with TMEM accumulators, TMA-staged Q/K/V tiles).
#include "prefill_common.cuh"

int pkv_prefill_tc_supported(const pkv::PrefillArgs& a, int head_dim) {
    (void)a;
    (void)head_dim;
    return PKV_ERR_UNSUPPORTED;
}

int pkv_launch_prefill_tc(pkv::PrefillArgs& a, cudaStream_t s) {
    (void)a;
    (void)s;
    return PKV_ERR_UNSUPPORTED;
}
