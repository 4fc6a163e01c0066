// qmv_matvec_cb2.cu -- instantiation of the decode matvec kernel for the CB2 format.
#include "qmv_matvec.cuh"

namespace qmv {

cudaError_t launch_matvec_cb2(const MatvecArgs& a) { return launch_matvec<CB2>(a); }

QMV_DEFINE_STATUS_ACCESSOR(status_cb2)

}  // namespace qmv
