// tc_bwd.cu -- tensor-core (tcgen05) PSA backward.
#include "psa_attn.h"
#include "psa_internal.h"

namespace psa {

bool tc_supported(int, int) { return false; }
size_t tc_workspace_bytes(long long, int, int) { return 0; }
int tc_bwd_launch(const BwdArgs&, std::string* err) {
    *err = "tensor-core backward not built";
    return PSA_ERR_UNSUPPORTED;
}
int tc_take_device_error(std::string*) { return 0; }

}  // namespace psa
