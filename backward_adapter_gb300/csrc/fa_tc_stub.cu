#include "fa_internal.h"
namespace fa {
bool tc_bwd_supported(const Shape&) { return false; }
cudaError_t tc_bwd(const BwdArgs&, const BwdPlan&, char*) { return cudaErrorNotSupported; }
}
