/* A plain C caller that runs kernels through libgdn.so: it allocates device buffers with cudaMalloc, copies the
 * inputs of a small fp32 workload in from host arrays, calls gdn_mtp_verify (with intermediate states) and
 * gdn_commit on a stream of its own, copies the results back and checks them against reference values that
 * the calling test computed with the CPU oracle and wrote next to the inputs.
 *
 *     verify_commit_from_c <dir>
 *
 * <dir> holds dims.txt ("B T HK HV DK DV num_slots") and raw little-endian arrays: q.bin k.bin v.bin a.bin
 * b.bin A_log.bin dt_bias.bin pool.bin (fp32), indices.bin accept_len.bin (int32), o_ref.bin (fp64, the
 * oracle's o) and cache_ref.bin (fp32, the oracle's intermediate states).  Exit status 0 = every check passed.
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

#define CUDA_OK(call)                                                                     \
    do {                                                                                  \
        cudaError_t e_ = (call);                                                          \
        if (e_ != cudaSuccess) {                                                          \
            fprintf(stderr, "%s failed: %s (line %d)\n", #call, cudaGetErrorString(e_), __LINE__); \
            exit(2);                                                                      \
        }                                                                                 \
    } while (0)

/* Reads <dir>/<name> whole; its size must be `bytes`. */
static void* read_array(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) {
        fprintf(stderr, "cannot open %s\n", path);
        exit(2);
    }
    void* buf = malloc(bytes ? bytes : 1);
    size_t got = fread(buf, 1, bytes, f);
    int extra = fgetc(f);
    fclose(f);
    if (got != bytes || extra != EOF) {
        fprintf(stderr, "%s: expected %zu bytes\n", path, bytes);
        exit(2);
    }
    return buf;
}

static void* to_device(const void* host, size_t bytes) {
    void* d = NULL;
    CUDA_OK(cudaMalloc(&d, bytes));
    CUDA_OK(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
    return d;
}

/* max |x - ref| <= rel * max |ref| over n values */
static void expect_close(const char* what, const float* x, const double* ref, size_t n, double rel) {
    double scale = 0.0, err = 0.0;
    for (size_t i = 0; i < n; ++i) scale = fmax(scale, fabs(ref[i]));
    for (size_t i = 0; i < n; ++i) {
        EXPECT(isfinite(x[i]), "%s[%zu] is not finite", what, i);
        err = fmax(err, fabs((double)x[i] - ref[i]));
    }
    EXPECT(err <= rel * scale, "%s: max|x - ref| = %.3e > %.1e * %.3e", what, err, rel, scale);
}

int main(int argc, char** argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: %s <dir>\n", argv[0]);
        return 2;
    }
    const char* dir = argv[1];
    char path[4096];
    snprintf(path, sizeof path, "%s/dims.txt", dir);
    FILE* f = fopen(path, "r");
    int B, T, HK, HV, DK, DV, S;
    if (!f || fscanf(f, "%d %d %d %d %d %d %d", &B, &T, &HK, &HV, &DK, &DV, &S) != 7) {
        fprintf(stderr, "cannot read %s\n", path);
        return 2;
    }
    fclose(f);

    const size_t n_qk = (size_t)B * T * HK * DK, n_v = (size_t)B * T * HV * DV, n_ab = (size_t)B * T * HV;
    const size_t n_state = (size_t)HV * DV * DK, n_pool = (size_t)S * n_state, n_cache = (size_t)B * T * n_state;
    float* q = read_array(dir, "q.bin", 4 * n_qk);
    float* k = read_array(dir, "k.bin", 4 * n_qk);
    float* v = read_array(dir, "v.bin", 4 * n_v);
    float* a = read_array(dir, "a.bin", 4 * n_ab);
    float* b = read_array(dir, "b.bin", 4 * n_ab);
    float* A_log = read_array(dir, "A_log.bin", 4 * (size_t)HV);
    float* dt_bias = read_array(dir, "dt_bias.bin", 4 * (size_t)HV);
    float* pool = read_array(dir, "pool.bin", 4 * n_pool);
    int32_t* idx = read_array(dir, "indices.bin", 4 * (size_t)B);
    int32_t* acc = read_array(dir, "accept_len.bin", 4 * (size_t)B);
    double* o_ref = read_array(dir, "o_ref.bin", 8 * n_v);
    float* cache_ref = read_array(dir, "cache_ref.bin", 4 * n_cache);

    cudaStream_t stream;
    CUDA_OK(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    void *dq = to_device(q, 4 * n_qk), *dk = to_device(k, 4 * n_qk), *dv = to_device(v, 4 * n_v);
    void *da = to_device(a, 4 * n_ab), *db = to_device(b, 4 * n_ab);
    float *dA = to_device(A_log, 4 * (size_t)HV), *ddt = to_device(dt_bias, 4 * (size_t)HV);
    void* dpool = to_device(pool, 4 * n_pool);
    int32_t *didx = to_device(idx, 4 * (size_t)B), *dacc = to_device(acc, 4 * (size_t)B);
    const int32_t zero = 0;
    int32_t* derr = to_device(&zero, 4);
    void *dout = NULL, *dcache = NULL;
    CUDA_OK(cudaMalloc(&dout, 4 * n_v));
    CUDA_OK(cudaMalloc(&dcache, 4 * n_cache));

    gdn_dims d;
    memset(&d, 0, sizeof d);
    d.B = B; d.T = T; d.HK = HK; d.HV = HV; d.DK = DK; d.DV = DV; d.num_slots = S;
    d.qkv_dtype = GDN_F32; d.state_dtype = GDN_F32; d.out_dtype = GDN_F32;
    d.scale = 1.0f; d.l2_eps = 1e-6f;
    gdn_status st = gdn_mtp_verify(&d, dq, dk, dv, da, db, dA, ddt, dpool, didx, dout, dcache, derr,
                                   (gdn_stream_t)stream);
    EXPECT(st == GDN_OK, "gdn_mtp_verify: %s", gdn_status_string(st));
    st = gdn_commit(&d, dpool, didx, dcache, dacc, derr, (gdn_stream_t)stream);
    EXPECT(st == GDN_OK, "gdn_commit: %s", gdn_status_string(st));

    float* o = malloc(4 * n_v);
    float* cache = malloc(4 * n_cache);
    float* pool_after = malloc(4 * n_pool);
    int32_t err = -1;
    CUDA_OK(cudaMemcpyAsync(o, dout, 4 * n_v, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaMemcpyAsync(cache, dcache, 4 * n_cache, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaMemcpyAsync(pool_after, dpool, 4 * n_pool, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaMemcpyAsync(&err, derr, 4, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaStreamSynchronize(stream));

    EXPECT(err == 0, "device error word %d", err);
    expect_close("o", o, o_ref, n_v, 1e-4);
    double* cref = malloc(8 * n_cache);
    for (size_t i = 0; i < n_cache; ++i) cref[i] = cache_ref[i];
    expect_close("intermediate_states", cache, cref, n_cache, 1e-4);
    /* commit: each active lane's slot holds cache[b, accept_len - 1] bit for bit; every other slot is unchanged */
    char* touched = calloc((size_t)S, 1);
    for (int lane = 0; lane < B; ++lane) {
        const int s = idx[lane], L = acc[lane];
        if (s < 0 || L < 1) continue;
        touched[s] = 1;
        EXPECT(memcmp(pool_after + (size_t)s * n_state, cache + ((size_t)lane * T + (L - 1)) * n_state,
                      4 * n_state) == 0,
               "slot %d differs from lane %d's cached state %d", s, lane, L - 1);
    }
    for (int s = 0; s < S; ++s)
        if (!touched[s])
            EXPECT(memcmp(pool_after + (size_t)s * n_state, pool + (size_t)s * n_state, 4 * n_state) == 0,
                   "uncommitted slot %d changed", s);

    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(da); cudaFree(db); cudaFree(dA); cudaFree(ddt);
    cudaFree(dpool); cudaFree(didx); cudaFree(dacc); cudaFree(derr); cudaFree(dout); cudaFree(dcache);
    cudaStreamDestroy(stream);
    free(q); free(k); free(v); free(a); free(b); free(A_log); free(dt_bias); free(pool); free(idx); free(acc);
    free(o_ref); free(cache_ref); free(o); free(cache); free(pool_after); free(cref); free(touched);
    if (failures == 0) printf("verify_commit_from_c: ok\n");
    return failures == 0 ? 0 : 1;
}
