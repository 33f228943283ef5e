// Instantiations of the two-channel selective-scan kernel with the chunk carry in one
// launch: bf16 and fp32 inputs, time-varying B and C, S = N states per lane.
#include "kernel_table.cuh"

namespace ssm {

template <typename IO, int S>
FusedInfo fused_info() {
  using Gm = FGeo<IO, S>;
  FusedInfo k;
  k.fn = scan_fused_kernel<IO, S>;
  k.nt = Gm::NT;
  k.ch = Gm::CH;
  k.cw = Gm::CW;
  k.t = Gm::T;
  k.smem = Gm::BYTES;
  return k;
}

FusedInfo lookup_fused(int io_bf16, int S) {
  if (io_bf16) {
    if (S == 8) return fused_info<BF16, 8>();
    if (S == 16) return fused_info<BF16, 16>();
  } else {
    if (S == 4) return fused_info<F32, 4>();
    if (S == 8) return fused_info<F32, 8>();
    if (S == 16) return fused_info<F32, 16>();
  }
  return FusedInfo();
}

}  // namespace ssm
