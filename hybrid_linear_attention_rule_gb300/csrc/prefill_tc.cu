// prefill_tc.cu -- tensor-core (tcgen05) chunked KDA prefill.  Placeholder:
// no shape is routed here yet.
#include "common.cuh"

namespace k3kda {

bool tc_prefill_supported(int in_bf16, int dk, int dv, int chunk) {
    (void)in_bf16; (void)dk; (void)dv; (void)chunk;
    return false;
}

size_t tc_prefill_workspace(int N, int H) { (void)N; (void)H; return 0; }

cudaError_t launch_prefill_tc(const PrefillArgs &a, const int32_t *order, cudaStream_t s) {
    (void)a; (void)order; (void)s;
    return cudaErrorNotSupported;
}

}  // namespace k3kda
