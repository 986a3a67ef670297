// Tensor-core (tcgen05 / TMEM / TMA) kernels of the hot path: host-side plan.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "kvc_internal.h"

namespace kvc {

// Tables the tensor-core kernels need, appended to the layer's parameter
// block by tc_prepare (as offsets) and turned into device pointers by tc_bind.
struct TcPlan {
  bool fetch_ready = false;
  bool append_ready = false;
};

kvc_status tc_prepare(const kvc_layer_desc& d, int d_in, int Hg, int nb, int r,
                      const std::vector<uint8_t>& bits, const std::vector<int16_t>& order,
                      const std::vector<int32_t>& n_kept, std::vector<uint8_t>& image,
                      TcPlan& plan);
void tc_bind(TcPlan& plan, uint8_t* block_base);
void tc_release(TcPlan& plan);

bool tc_append_ok(const TcPlan& plan, const Params& p, const AppendArgs& a);
bool tc_fetch_ok(const TcPlan& plan, const Params& p, const FetchArgs& f);
cudaError_t launch_append_tc(const TcPlan& plan, const Params& p, const AppendArgs& a,
                             cudaStream_t s, int* nk);
cudaError_t launch_fetch_tc(const TcPlan& plan, const Params& p, const FetchArgs& f,
                            cudaStream_t s, int* nk);

}  // namespace kvc
