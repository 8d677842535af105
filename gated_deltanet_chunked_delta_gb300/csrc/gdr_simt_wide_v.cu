// gdr_simt_wide_v.cu -- the CUDA-core path at V in {192, 256} with K in {64,
// 128}.  Kernels: gdr_simt_kernels.cuh.
#include "gdr_simt_kernels.cuh"

namespace gdr {

int simt_fwd_wide_v(const Params &p, int in_f32, int o_f32, int use_cp, cudaStream_t st) {
    if (p.K == 64 && p.V == 192) return fwd_sized<64, 192>(p, in_f32, o_f32, use_cp, st);
    if (p.K == 64 && p.V == 256) return fwd_sized<64, 256>(p, in_f32, o_f32, use_cp, st);
    if (p.K == 128 && p.V == 192) return fwd_sized<128, 192>(p, in_f32, o_f32, use_cp, st);
    if (p.K == 128 && p.V == 256) return fwd_sized<128, 256>(p, in_f32, o_f32, use_cp, st);
    return 1;
}

int simt_bwd_wide_v(const Params &p, int in_f32, int use_cp, cudaStream_t st) {
    if (p.K == 64 && p.V == 192) return bwd_sized<64, 192>(p, in_f32, use_cp, st);
    if (p.K == 64 && p.V == 256) return bwd_sized<64, 256>(p, in_f32, use_cp, st);
    if (p.K == 128 && p.V == 192) return bwd_sized<128, 192>(p, in_f32, use_cp, st);
    if (p.K == 128 && p.V == 256) return bwd_sized<128, 256>(p, in_f32, use_cp, st);
    return 1;
}

unsigned simt_wide_v_take_status(cudaStream_t st) { return take_status(st); }

}  // namespace gdr
