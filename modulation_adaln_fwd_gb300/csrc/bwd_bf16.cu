// bwd_bf16.cu -- bf16 instantiations of the pipelined backward kernels.
#include "bwd_ring.cuh"

namespace adaln {

cudaError_t bwd_ring_bf16(const void *x, const float *mean, const float *rstd, const void *scale,
                          const void *dy, void *dx, float *partial, int *status,
                          const Segments &sg, const Chunking &ch, int D, const void *gate,
                          cudaStream_t s) {
    return bwd_dispatch<__nv_bfloat16>(x, mean, rstd, scale, dy, dx, partial, status, sg, ch, D,
                                       gate, s);
}

cudaError_t gate_bwd_ring_bf16(const void *dout, const void *z, const void *gate, void *dz,
                               float *partial, int *status, const Segments &sg,
                               const Chunking &ch, int D, cudaStream_t s) {
    return gate_bwd_dispatch<__nv_bfloat16>(dout, z, gate, dz, partial, status, sg, ch, D, s);
}

bool bwd_ring_fits(DType dt, int64_t D, bool gate) {
    DeviceInfo di;
    if (device_info(di) != cudaSuccess) return false;
    if (D <= 0 || D > (int64_t)1 << 20) return false;
    RingGeom g;
    return dt == DType::BF16 ? ring_geometry((int)D, 2, 8, di, g, !gate)
                             : ring_geometry((int)D, 4, 4, di, g, !gate);
}

int bwd_ring_ctas_per_sm(DType dt, int64_t D, bool gate) {
    DeviceInfo di;
    if (device_info(di) != cudaSuccess) return 1;
    if (D <= 0 || D > (int64_t)1 << 20) return 1;
    return dt == DType::BF16 ? ctas_per_sm<__nv_bfloat16>((int)D, gate, di)
                             : ctas_per_sm<float>((int)D, gate, di);
}

}  // namespace adaln
