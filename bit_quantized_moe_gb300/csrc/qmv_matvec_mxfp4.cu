// qmv_matvec_mxfp4.cu -- instantiation of the decode matvec kernel for the MXFP4 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_mxfp4(const MatvecArgs& a) { return launch_matvec<MXFP4>(a); }

QMV_DEFINE_STATUS_ACCESSOR(status_mxfp4)

}  // namespace qmv
