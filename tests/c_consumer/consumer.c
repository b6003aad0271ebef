/*
 * A plain C99 consumer of the library's C ABI (include/gated_act.h): no
 * Python, no PyTorch.  It reads bf16 rows from a file, runs
 * gelu_and_mul_sparse, gelu_and_mul_sparse_ws and silu_and_mul on device
 * buffers it allocates with the CUDA runtime, and writes the results back to
 * files for the test to compare with the oracle.
 *
 *   consumer <T> <d> <z> <gelu_in> <gelu_out> <gelu_ws_out> <M> <silu_in> <silu_out>
 *
 * Exit status 0 on success; otherwise it prints the failing call and the
 * library's status text.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "gated_act.h"

static int fail(const char *what, int status) {
    fprintf(stderr, "%s: status %d: %s\n", what, status, gated_act_status_string(status));
    return 1;
}

static int cuda_fail(const char *what, cudaError_t e) {
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return 1;
}

static void *read_file(const char *path, size_t bytes) {
    FILE *f = fopen(path, "rb");
    void *p = malloc(bytes ? bytes : 1);
    if (!f || !p || fread(p, 1, bytes, f) != bytes) {
        if (f)
            fclose(f);
        free(p);
        return NULL;
    }
    fclose(f);
    return p;
}

static int write_file(const char *path, const void *p, size_t bytes) {
    FILE *f = fopen(path, "wb");
    if (!f)
        return 1;
    const int bad = fwrite(p, 1, bytes, f) != bytes;
    return fclose(f) != 0 || bad;
}

/* Copy `in_bytes` to the device, run `call`, copy `out_bytes` back. */
typedef int (*op_fn)(void *out, const void *in, void *ctx);

static int run_op(const char *name, op_fn call, void *ctx, const void *host_in, size_t in_bytes,
                  void *host_out, size_t out_bytes) {
    void *din = NULL, *dout = NULL;
    cudaError_t e = cudaMalloc(&din, in_bytes);
    if (e == cudaSuccess)
        e = cudaMalloc(&dout, out_bytes);
    if (e == cudaSuccess)
        e = cudaMemcpy(din, host_in, in_bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess)
        return cuda_fail(name, e);
    const int rc = call(dout, din, ctx);
    if (rc != GATED_ACT_OK)
        return fail(name, rc);
    e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(host_out, dout, out_bytes, cudaMemcpyDeviceToHost);
    cudaFree(din);
    cudaFree(dout);
    return e == cudaSuccess ? 0 : cuda_fail(name, e);
}

struct gelu_args {
    int64_t T, d;
    double z;
    void *workspace;
};

static int call_gelu(void *out, const void *in, void *ctx) {
    const struct gelu_args *a = (const struct gelu_args *)ctx;
    return gelu_and_mul_sparse(out, in, a->T, a->d, 2 * a->d, a->z, 0);
}

static int call_gelu_ws(void *out, const void *in, void *ctx) {
    const struct gelu_args *a = (const struct gelu_args *)ctx;
    return gelu_and_mul_sparse_ws(out, in, a->T, a->d, 2 * a->d, a->z, GATED_ACT_BF16,
                                  GATED_ACT_VARIANT_TMA_ROWS, 0, a->workspace, 0);
}

static int call_silu(void *out, const void *in, void *ctx) {
    const int64_t *md = (const int64_t *)ctx;
    return silu_and_mul(out, in, md[0], md[1], 0);
}

int main(int argc, char **argv) {
    if (argc != 10) {
        fprintf(stderr, "usage: %s T d z gelu_in gelu_out gelu_ws_out M silu_in silu_out\n",
                argv[0]);
        return 2;
    }
    struct gelu_args g;
    g.T = strtoll(argv[1], NULL, 10);
    g.d = strtoll(argv[2], NULL, 10);
    g.z = strtod(argv[3], NULL);
    g.workspace = NULL;
    int64_t silu_md[2];
    silu_md[0] = strtoll(argv[7], NULL, 10);
    silu_md[1] = 768;

    const size_t gin = (size_t)(g.T * 2 * g.d) * 2, gout = (size_t)(g.T * g.d) * 2;
    const size_t sin = (size_t)(silu_md[0] * 2 * silu_md[1]) * 2;
    const size_t sout = (size_t)(silu_md[0] * silu_md[1]) * 2;
    void *x = read_file(argv[4], gin), *s = read_file(argv[8], sin);
    void *y = malloc(gout), *y_ws = malloc(gout), *t = malloc(sout);
    if (!x || !s || !y || !y_ws || !t) {
        fprintf(stderr, "cannot read the inputs\n");
        return 1;
    }

    /* a zeroed device workspace, as the header asks */
    cudaError_t e = cudaMalloc(&g.workspace, gelu_and_mul_sparse_workspace_bytes());
    if (e == cudaSuccess)
        e = cudaMemset(g.workspace, 0, gelu_and_mul_sparse_workspace_bytes());
    if (e != cudaSuccess)
        return cuda_fail("workspace", e);

    if (run_op("gelu_and_mul_sparse", call_gelu, &g, x, gin, y, gout) ||
        run_op("gelu_and_mul_sparse_ws", call_gelu_ws, &g, x, gin, y_ws, gout) ||
        run_op("silu_and_mul", call_silu, silu_md, s, sin, t, sout))
        return 1;

    /* the workspace is left zeroed */
    uint64_t counters[2] = {1, 1};
    e = cudaMemcpy(counters, g.workspace, sizeof counters, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail("workspace read-back", e);
    if (counters[0] != 0 || counters[1] != 0) {
        fprintf(stderr, "workspace not left zeroed\n");
        return 1;
    }
    cudaFree(g.workspace);

    /* a bad call is refused with a status, and launches nothing */
    const int rc = gelu_and_mul_sparse(y, x, g.T, g.d, g.d, g.z, 0);   /* row_stride < 2d */
    if (rc != GATED_ACT_ERR_STRIDE)
        return fail("row_stride < 2d was not refused", rc);

    if (write_file(argv[5], y, gout) || write_file(argv[6], y_ws, gout) ||
        write_file(argv[9], t, sout)) {
        fprintf(stderr, "cannot write the outputs\n");
        return 1;
    }
    free(x);
    free(s);
    free(y);
    free(y_ws);
    free(t);
    printf("ok\n");
    return 0;
}
