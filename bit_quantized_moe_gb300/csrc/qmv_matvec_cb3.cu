// qmv_matvec_cb3.cu -- instantiation of the decode matvec kernel for the CB3 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_cb3(const MatvecArgs& a) { return launch_matvec<CB3>(a); }

QMV_DEFINE_STATUS_ACCESSOR(status_cb3)

}  // namespace qmv
