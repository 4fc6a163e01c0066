// qmv_matvec_mxfp8.cu -- instantiation of the decode matvec kernel for the MXFP8 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_mxfp8(const MatvecArgs& a) { return launch_matvec<MXFP8>(a); }

QMV_DEFINE_STATUS_ACCESSOR(status_mxfp8)

}  // namespace qmv
