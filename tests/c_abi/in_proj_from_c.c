/* A plain C caller of the in_proj projection with its conv1d epilogue: it allocates device buffers with cudaMalloc,
 * copies a small workload in from host arrays, calls gdn_in_proj_conv (decode rows: the convolution state written
 * back) on a stream of its own, copies the results back and checks them against reference values that the calling
 * test computed with the CPU oracle and wrote next to the inputs.
 *
 *     in_proj_from_c <dir>
 *
 * <dir> holds dims.txt ("B T H HK HV DK DV K num_slots") and raw little-endian arrays: x.bin, W.bin and state.bin
 * (bf16 bit patterns), conv_w.bin and conv_b.bin (fp32), indices.bin (int32), out_ref.bin (fp64 [B, T, C]: the
 * oracle's outputs in W's channel order) and state_ref.bin (bf16 bits: the oracle's state after the call).
 * Outputs are fp32.  Exit status 0 = every check passed.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "gdn.h"

static int failures = 0;

#define EXPECT(cond, ...)                                         \
    do {                                                          \
        if (!(cond)) {                                            \
            fprintf(stderr, "FAILED (line %d): ", __LINE__);      \
            fprintf(stderr, __VA_ARGS__);                         \
            fprintf(stderr, "\n");                                \
            ++failures;                                           \
        }                                                         \
    } while (0)

#define CUDA_OK(call)                                                                                  \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess) {                                                                       \
            fprintf(stderr, "%s failed: %s (line %d)\n", #call, cudaGetErrorString(e_), __LINE__);     \
            exit(2);                                                                                   \
        }                                                                                              \
    } while (0)

static void* read_file(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) {
        fprintf(stderr, "cannot open %s\n", path);
        exit(2);
    }
    void* buf = malloc(bytes ? bytes : 1);
    if (fread(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "short read of %s\n", path);
        exit(2);
    }
    fclose(f);
    return buf;
}

static void* to_device(const void* host, size_t bytes) {
    void* d = NULL;
    CUDA_OK(cudaMalloc(&d, bytes ? bytes : 16));
    if (bytes) CUDA_OK(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
    return d;
}

static double bf16_to_double(uint16_t h) {
    uint32_t w = (uint32_t)h << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

int main(int argc, char** argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: %s <dir>\n", argv[0]);
        return 2;
    }
    const char* dir = argv[1];
    char dims_path[4096];
    snprintf(dims_path, sizeof dims_path, "%s/dims.txt", dir);
    FILE* df = fopen(dims_path, "r");
    if (!df) return 2;
    gdn_conv_dims d;
    memset(&d, 0, sizeof d);
    if (fscanf(df, "%d %d %d %d %d %d %d %d %d", &d.B, &d.T, &d.H, &d.HK, &d.HV, &d.DK, &d.DV, &d.K, &d.num_slots) !=
        9)
        return 2;
    fclose(df);
    d.conv_dtype = GDN_BF16;
    d.out_dtype = GDN_F32;
    d.silu = 1;
    const size_t rows = (size_t)d.B * d.T;
    const size_t qk = (size_t)d.HK * d.DK, vz = (size_t)d.HV * d.DV;
    const size_t Cc = 2 * qk + vz, C = Cc + vz + 2 * (size_t)d.HV;
    const size_t state_elems = (size_t)d.num_slots * (d.K - 1) * Cc;

    uint16_t* x = read_file(dir, "x.bin", rows * d.H * 2);
    uint16_t* W = read_file(dir, "W.bin", C * d.H * 2);
    float* conv_w = read_file(dir, "conv_w.bin", Cc * d.K * 4);
    float* conv_b = read_file(dir, "conv_b.bin", Cc * 4);
    uint16_t* state = read_file(dir, "state.bin", state_elems * 2);
    int32_t* idx = read_file(dir, "indices.bin", (size_t)d.B * 4);
    double* out_ref = read_file(dir, "out_ref.bin", rows * C * 8);
    uint16_t* state_ref = read_file(dir, "state_ref.bin", state_elems * 2);

    void* dx = to_device(x, rows * d.H * 2);
    void* dW = to_device(W, C * d.H * 2);
    void* dw = to_device(conv_w, Cc * d.K * 4);
    void* db = to_device(conv_b, Cc * 4);
    void* dstate = to_device(state, state_elems * 2);
    void* didx = to_device(idx, (size_t)d.B * 4);
    const size_t sizes[6] = {rows * qk, rows * qk, rows * vz, rows * vz, rows * d.HV, rows * d.HV};
    void* dout[6];
    for (int i = 0; i < 6; ++i) {
        CUDA_OK(cudaMalloc(&dout[i], sizes[i] * 4));
        CUDA_OK(cudaMemset(dout[i], 0xFF, sizes[i] * 4));  /* NaN canaries */
    }
    int32_t* derr = NULL;
    CUDA_OK(cudaMalloc((void**)&derr, 4));
    CUDA_OK(cudaMemset(derr, 0, 4));
    gdn_in_proj_out out = {dout[0], dout[1], dout[2], dout[3], dout[4], dout[5]};

    cudaStream_t stream;
    CUDA_OK(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    gdn_status s = gdn_in_proj_conv(&d, dx, dW, dw, db, dstate, didx, 1, &out, NULL, derr, (gdn_stream_t)stream);
    EXPECT(s == GDN_OK, "gdn_in_proj_conv: %s", gdn_status_string(s));
    CUDA_OK(cudaStreamSynchronize(stream));

    int32_t err_word = -1;
    CUDA_OK(cudaMemcpy(&err_word, derr, 4, cudaMemcpyDeviceToHost));
    EXPECT(err_word == 0, "error word %d", err_word);

    /* outputs in W's channel order: q | k | v | z | b | a */
    float* got[6];
    for (int i = 0; i < 6; ++i) {
        got[i] = malloc(sizes[i] * 4);
        CUDA_OK(cudaMemcpy(got[i], dout[i], sizes[i] * 4, cudaMemcpyDeviceToHost));
    }
    const size_t width[6] = {qk, qk, vz, vz, (size_t)d.HV, (size_t)d.HV};
    double worst = 0.0;
    for (int b = 0; b < d.B; ++b) {
        const int active = idx[b] >= 0;
        for (int t = 0; t < d.T; ++t) {
            const size_t row = (size_t)b * d.T + t;
            size_t c0 = 0;
            for (int i = 0; i < 6; ++i) {
                for (size_t c = 0; c < width[i]; ++c) {
                    const float v = got[i][row * width[i] + c];
                    if (!active) {
                        EXPECT(isnan(v), "padded lane %d row %d: output %d written", b, t, i);
                        continue;
                    }
                    const double diff = fabs((double)v - out_ref[row * C + c0 + c]);
                    if (diff > worst) worst = diff;
                }
                c0 += width[i];
            }
        }
    }
    /* values are O(1): the stored state rounds each product to bf16 (1 ulp = 2^-8 relative at most) */
    EXPECT(worst <= 2e-2, "outputs: max |gpu - oracle| = %.3e", worst);

    uint16_t* state_got = malloc(state_elems * 2);
    CUDA_OK(cudaMemcpy(state_got, dstate, state_elems * 2, cudaMemcpyDeviceToHost));
    size_t differ = 0;
    for (size_t i = 0; i < state_elems; ++i) {
        const double a = bf16_to_double(state_got[i]), r = bf16_to_double(state_ref[i]);
        if (state_got[i] != state_ref[i]) ++differ;
        EXPECT(fabs(a - r) <= ldexp(fabs(r), -7) + 1e-30, "state element %zu: %g against %g", i, a, r);
    }
    EXPECT(differ * 20 <= state_elems, "state: %zu of %zu elements differ from the oracle's bits", differ,
           state_elems);

    CUDA_OK(cudaStreamDestroy(stream));
    if (failures == 0) printf("in_proj_from_c: ok (max output difference %.3e)\n", worst);
    return failures == 0 ? 0 : 1;
}
