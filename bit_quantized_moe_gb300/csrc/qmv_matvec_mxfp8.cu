// qmv_matvec_mxfp8.cu -- instantiation of the decode matvec kernel for the MXFP8 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_mxfp8(const MatvecArgs& a) { return launch_matvec<MXFP8>(a); }
cudaError_t launch_chunk_rate_mxfp8(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                  int64_t* threads, cudaStream_t s) {
  return launch_chunk_rate<MXFP8>(nv, ctas_per_sm, iters, sink, weights, threads, s);
}

QMV_DEFINE_STATUS_ACCESSOR(status_mxfp8)
QMV_DEFINE_PHASE_ACCESSOR(phase_mxfp8)

}  // namespace qmv
