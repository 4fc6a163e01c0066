// qmv_matvec_cb2.cu -- instantiation of the decode matvec kernel for the CB2 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_cb2(const MatvecArgs& a) { return launch_matvec<CB2>(a); }
cudaError_t launch_chunk_rate_cb2(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                  int64_t* threads, cudaStream_t s) {
  return launch_chunk_rate<CB2>(nv, ctas_per_sm, iters, sink, weights, threads, s);
}

QMV_DEFINE_STATUS_ACCESSOR(status_cb2)
QMV_DEFINE_PHASE_ACCESSOR(phase_cb2)

}  // namespace qmv
