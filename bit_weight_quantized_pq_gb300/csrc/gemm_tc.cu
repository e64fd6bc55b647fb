// Prefill GEMM (M >= 17): placeholder until the tcgen05 kernel lands.
#include "pq_internal.cuh"

namespace pq {

bool gemm_supported(const pq_desc&) { return false; }
void plan_gemm(const pq_prepared*, int, pq_plan_info* info) { info->variant = PQ_VARIANT_W4_GEMM; }
int32_t gemm_init(pq_prepared*) { return PQ_OK; }
void gemm_free(pq_prepared*) {}
cudaError_t launch_w4_gemm(const pq_prepared*, const void*, void*, int, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_w2_gemm(const pq_prepared*, const void*, void*, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace pq
