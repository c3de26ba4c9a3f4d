// bwd_f32.cu -- fp32 instantiations of the pipelined backward kernels.
#include "bwd_ring.cuh"

namespace adaln {

cudaError_t bwd_ring_f32(const void *x, const float *mean, const float *rstd, const void *scale,
                         const void *dy, void *dx, float *partial, int *status,
                         const Segments &sg, const Chunking &ch, int D, const void *gate,
                         cudaStream_t s) {
    return bwd_dispatch<float>(x, mean, rstd, scale, dy, dx, partial, status, sg, ch, D, gate, s);
}

cudaError_t gate_bwd_ring_f32(const void *dout, const void *z, const void *gate, void *dz,
                              float *partial, int *status, const Segments &sg,
                              const Chunking &ch, int D, cudaStream_t s) {
    return gate_bwd_dispatch<float>(dout, z, gate, dz, partial, status, sg, ch, D, s);
}

}  // namespace adaln
