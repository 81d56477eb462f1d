// layer_front: the kernel that runs before the QKV front in the first decoder
// layer (included by qkv_front.cu: one translation unit).
//
// Source: page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.
// boundary.layer_front", class LayerFront: run(x, stream, out, aux) writes
// stream = x as FP32 (the residual stream), aux = stream when the layer keeps
// one, and out = the layer's pre-QKV RMS norm of the stream in BF16 — the x
// the QKV front reads.  x is BF16 or FP32 [rows, 8192].  With PDL the page's
// kernel releases its dependents right after its own wait, and the QKV front
// waits for this grid before it reads out (page layer_front, module
// docstring).  This one releases them at entry, before its wait: the front
// reads only its weights before its own wait, which covers this grid and so,
// transitively, the kernel before it; releasing early lets the next front's
// CTAs take SMs the moment the previous front's CTAs leave, so its weight
// stream also overlaps the previous front's tail, not only this kernel.
//
// The norm (the page names it, not its formula; the plainest reading): over
// the whole row, r = 1 / sqrt(mean_j s_j^2 + eps); out_j = bf16((s_j r) w_j)
// with the BF16 weight widened to FP32, or bf16(s_j r) without a weight.
//
// One CTA per row, 256 threads, each owning four 8-element chunks
// (chunk k: elements 2048 k + 8 tid .. + 7): 16-byte loads and stores,
// coalesced across the CTA.  The sum of squares is sequential per thread,
// then a warp butterfly, then the 8 warp sums in warp order: deterministic.

namespace qkvf {

constexpr int kLfThreads = 256;
constexpr int kLfMaxRows = 1 << 20;

struct LayerFrontParams {
    const void *x;
    const uint16_t *weight;   // [8192] bf16 bits, or null (weightless)
    float *stream;
    float *aux;               // or null
    uint16_t *out;
    float eps;
    int x_is_f32;
};

__global__ void __launch_bounds__(kLfThreads) layer_front_kernel(const LayerFrontParams p)
{
    __shared__ float warp_ss[kLfThreads / 32];
    // release dependents at once: until their own wait they read only weights
    if (threadIdx.x == 0) griddep_launch_dependents();
    griddep_wait();   // x is written by the kernel before this one
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t row = (size_t)blockIdx.x * kHidden;
    float v[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const size_t e = row + (size_t)k * (kLfThreads * 8) + 8 * tid;
        if (p.x_is_f32) {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(p.x) + e);
            const float4 a = src[0], b = src[1];
            v[k][0] = a.x; v[k][1] = a.y; v[k][2] = a.z; v[k][3] = a.w;
            v[k][4] = b.x; v[k][5] = b.y; v[k][6] = b.z; v[k][7] = b.w;
        } else {
            const uint4 w = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.x) + e);
            const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&w4[j]);
                v[k][2 * j] = __low2float(pr);
                v[k][2 * j + 1] = __high2float(pr);
            }
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) ss = __fadd_rn(ss, __fmul_rn(v[k][j], v[k][j]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    if (lane == 0) warp_ss[warp] = ss;
    __syncthreads();
    float total = warp_ss[0];
#pragma unroll
    for (int w = 1; w < kLfThreads / 32; ++w) total = __fadd_rn(total, warp_ss[w]);
    const float ms = __fmul_rn(total, 1.0f / (float)kHidden);   // exact: a power of two
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, p.eps)));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const size_t col = (size_t)k * (kLfThreads * 8) + 8 * tid;
        const size_t e = row + col;
        float4 *s4 = reinterpret_cast<float4 *>(p.stream + e);
        s4[0] = make_float4(v[k][0], v[k][1], v[k][2], v[k][3]);
        s4[1] = make_float4(v[k][4], v[k][5], v[k][6], v[k][7]);
        if (p.aux) {
            float4 *a4 = reinterpret_cast<float4 *>(p.aux + e);
            a4[0] = s4[0];
            a4[1] = s4[1];
        }
        float wv[8];
        if (p.weight) {
            const uint4 w = *reinterpret_cast<const uint4 *>(p.weight + col);
            const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&w4[j]);
                wv[2 * j] = __low2float(pr);
                wv[2 * j + 1] = __high2float(pr);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float y0 = __fmul_rn(v[k][2 * j], r), y1 = __fmul_rn(v[k][2 * j + 1], r);
            if (p.weight) {
                y0 = __fmul_rn(y0, wv[2 * j]);
                y1 = __fmul_rn(y1, wv[2 * j + 1]);
            }
            o[j] = pack_bf16x2(__float2bfloat16_rn(y0), __float2bfloat16_rn(y1));
        }
        *reinterpret_cast<uint4 *>(p.out + e) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

const char *check_layer_front_args(const void *x, int x_is_f32, const uint16_t *weight,
                                   float *stream, float *aux, uint16_t *out, int rows, float eps,
                                   int *code)
{
    *code = QKVF_ERR_TOKENS;
    if (rows < 0 || rows > kLfMaxRows) return "rows must be 0..1048576";
    *code = QKVF_ERR_ARG;
    if (x_is_f32 != 0 && x_is_f32 != 1) return "x_is_f32 must be 0 or 1";
    if (!(eps > 0.f) || eps > 1.f) return "eps must be in (0, 1]";
    *code = QKVF_OK;
    if (rows == 0) return nullptr;
    *code = QKVF_ERR_NULL;
    if (!x || !stream || !out) return "x, stream and out are required";
    *code = QKVF_ERR_ALIGN;
    if (!aligned(x, 16) || !aligned(stream, 16) || !aligned(out, 16) ||
        (aux && !aligned(aux, 16)) || (weight && !aligned(weight, 16)))
        return "every array must be 16-byte aligned";
    *code = QKVF_ERR_ARG;
    const size_t n = (size_t)rows * kHidden;
    const size_t x_b = n * (x_is_f32 ? 4 : 2), s_b = n * 4, o_b = n * 2, w_b = kHidden * 2;
    const void *outs[] = {stream, aux, out};
    const size_t out_b[] = {s_b, aux ? s_b : 0, o_b};
    for (int i = 0; i < 3; ++i) {
        if (overlap(x, x_b, outs[i], out_b[i]) || (weight && overlap(weight, w_b, outs[i], out_b[i])))
            return "an input overlaps an output";
        for (int j = i + 1; j < 3; ++j)
            if (overlap(outs[i], out_b[i], outs[j], out_b[j])) return "outputs overlap";
    }
    *code = QKVF_OK;
    return nullptr;
}

}  // namespace qkvf

extern "C" {

int layer_front(const void *x, int x_is_f32, const uint16_t *weight, float *stream, float *aux,
                uint16_t *out, int rows, float eps, void *cuda_stream)
{
    int code;
    if (qkvf::check_layer_front_args(x, x_is_f32, weight, stream, aux, out, rows, eps, &code))
        return code;
    if (rows == 0) return QKVF_OK;
    qkvf::DeviceState *d;
    const int rc = qkvf::probe_device(&d);
    if (rc != QKVF_OK) return rc;
    qkvf::LayerFrontParams prm;
    prm.x = x;
    prm.weight = weight;
    prm.stream = stream;
    prm.aux = aux;
    prm.out = out;
    prm.eps = eps;
    prm.x_is_f32 = x_is_f32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows, 1, 1);
    cfg.blockDim = dim3(qkvf::kLfThreads, 1, 1);
    cfg.stream = (cudaStream_t)cuda_stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = qkvf::g_pdl ? 1 : 0;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, qkvf::layer_front_kernel, prm) != cudaSuccess) {
        (void)cudaGetLastError();
        return QKVF_ERR_CUDA;
    }
    return QKVF_OK;
}

}  // extern "C"
