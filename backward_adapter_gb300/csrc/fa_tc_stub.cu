#include "fa_internal.h"
namespace fa {
bool tc_supported(const Shape&) { return false; }
int tc_fwd_kv_splits(const Shape&) { return 1; }
cudaError_t tc_fwd(const FwdArgs&, const FwdPlan&, char*) { return cudaErrorNotSupported; }
cudaError_t tc_bwd(const BwdArgs&, const BwdPlan&, char*) { return cudaErrorNotSupported; }
}
