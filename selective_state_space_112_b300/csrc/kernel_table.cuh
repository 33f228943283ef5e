// Kernel lookup for the tiled selective-scan kernel: one entry per (io dtype, B/C
// layout, input-term form, pass (0: chunk aggregates, 1: output, 2: the whole call in
// one launch), states per lane S, lanes per channel G).  The
// instantiations are spread over ten translation units
// (kernels_<io>_<layout>[_zoh|_conv].cu) so that they build in parallel.
#pragma once

#include "scan_tile.cuh"

namespace ssm {

typedef void (*TileFn)(TmaMaps, ScanParams);

struct KernelInfo {
  TileFn fn = nullptr;
  int nt = 0;    // threads per CTA
  int ch = 0;    // channels per CTA
  int t = 0;     // steps per tile
  int smem = 0;  // dynamic shared memory bytes
};

// (S, G) pairs built: S states per lane in {2, 4, 8, 16}, G lanes per channel in
// {1, 2, 4}, S * G (the padded state count) in {2, ..., 64}.
#define SSM_FOR_EACH_SG(X) \
  X(2, 1) X(4, 1) X(2, 2) X(8, 1) X(4, 2) X(2, 4) X(16, 1) X(8, 2) X(4, 4) \
  X(16, 2) X(8, 4) X(16, 4)

template <typename IO, int S, int G, bool LTI, int PASS, int VAR>
KernelInfo kernel_info() {
  using Gm = Geo<IO, S, G>;
  KernelInfo k;
  if constexpr (PASS == 2) k.fn = scan_onelaunch_kernel<IO, S, G, LTI, VAR>;
  else k.fn = scan_tile_kernel<IO, S, G, LTI, PASS, VAR>;
  k.nt = Gm::NT;
  k.ch = Gm::CH;
  k.t = Gm::T;
  k.smem = Gm::BYTES;
  return k;
}

template <typename IO, bool LTI, int PASS, int VAR>
KernelInfo pick_sg(int S, int G) {
#define SSM_CASE(s_, g_) \
  if (S == s_ && G == g_) return kernel_info<IO, s_, g_, LTI, PASS, VAR>();
  SSM_FOR_EACH_SG(SSM_CASE)
#undef SSM_CASE
  return KernelInfo();
}

template <typename IO, bool LTI, int VAR>
KernelInfo lookup_impl(int S, int G, int pass) {
  if (pass == 2) return pick_sg<IO, LTI, 2, VAR>(S, G);
  return pass ? pick_sg<IO, LTI, 1, VAR>(S, G) : pick_sg<IO, LTI, 0, VAR>(S, G);
}

// Defined in kernels_<io>_<layout>[_zoh].cu.
KernelInfo lookup_f32_tv(int S, int G, int pass);
KernelInfo lookup_f32_lti(int S, int G, int pass);
KernelInfo lookup_bf16_tv(int S, int G, int pass);
KernelInfo lookup_bf16_lti(int S, int G, int pass);
KernelInfo lookup_f32_tv_zoh(int S, int G, int pass);
KernelInfo lookup_f32_lti_zoh(int S, int G, int pass);
KernelInfo lookup_bf16_tv_zoh(int S, int G, int pass);
KernelInfo lookup_bf16_lti_zoh(int S, int G, int pass);
KernelInfo lookup_f32_tv_conv(int S, int G, int pass);
KernelInfo lookup_bf16_tv_conv(int S, int G, int pass);

// Recurrent step kernel (sequence length 1), step_kernel.cu: G threads per channel of
// 4 states each, G in {1, 2, 4, 8, 16}.
KernelInfo lookup_step(int io_bf16, bool lti, int G, bool conv);

}  // namespace ssm
