// qmv_matvec_cb4.cu -- instantiation of the decode matvec kernel for the CB4 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_cb4(const MatvecArgs& a) { return launch_matvec<CB4>(a); }

QMV_DEFINE_STATUS_ACCESSOR(status_cb4)

}  // namespace qmv
