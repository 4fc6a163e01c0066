// qmv_matvec_mxfp4.cu -- instantiation of the decode matvec kernel for the MXFP4 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_mxfp4(const MatvecArgs& a) { return launch_matvec<MXFP4>(a); }
cudaError_t launch_chunk_rate_mxfp4(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                  int64_t* threads, cudaStream_t s) {
  return launch_chunk_rate<MXFP4>(nv, ctas_per_sm, iters, sink, weights, threads, s);
}

QMV_DEFINE_STATUS_ACCESSOR(status_mxfp4)
QMV_DEFINE_PHASE_ACCESSOR(phase_mxfp4)

}  // namespace qmv
