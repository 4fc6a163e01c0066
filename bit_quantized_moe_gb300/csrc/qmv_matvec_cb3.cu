// qmv_matvec_cb3.cu -- instantiation of the decode matvec kernel for the CB3 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_cb3(const MatvecArgs& a) { return launch_matvec<CB3>(a); }
cudaError_t launch_chunk_rate_cb3(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                  int64_t* threads, cudaStream_t s) {
  return launch_chunk_rate<CB3>(nv, ctas_per_sm, iters, sink, weights, threads, s);
}

QMV_DEFINE_STATUS_ACCESSOR(status_cb3)
QMV_DEFINE_PHASE_ACCESSOR(phase_cb3)

}  // namespace qmv
