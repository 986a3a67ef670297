// Tensor-core kernels of the hot path (sm_103a).
#include "kvc_tc.h"

namespace kvc {

kvc_status tc_prepare(const kvc_layer_desc&, int, int, int, int, const std::vector<uint8_t>&,
                      const std::vector<int16_t>&, const std::vector<int32_t>&,
                      std::vector<uint8_t>&, TcPlan& plan) {
  plan = TcPlan{};
  return KVC_OK;
}
void tc_bind(TcPlan&, uint8_t*) {}
void tc_release(TcPlan&) {}
bool tc_append_ok(const TcPlan& plan, const Params&, const AppendArgs&) { return plan.append_ready; }
bool tc_fetch_ok(const TcPlan& plan, const Params&, const FetchArgs&) { return plan.fetch_ready; }
cudaError_t launch_append_tc(const TcPlan&, const Params&, const AppendArgs&, cudaStream_t, int*) {
  return cudaErrorNotSupported;
}
cudaError_t launch_fetch_tc(const TcPlan&, const Params&, const FetchArgs&, cudaStream_t, int*) {
  return cudaErrorNotSupported;
}

}  // namespace kvc
