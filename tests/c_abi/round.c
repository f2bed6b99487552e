/*
 * A C caller of libps with no Python: one PreSTO round (scoring, suffix sums,
 * log A and the walk; PreSTO section 3.2 steps (2)-(3)) through the C ABI of
 * include/ps.h.  It reads one subtree batch from raw files, copies it to the
 * device with the CUDA runtime, calls ps_score_walk_subtree on the legacy
 * default stream, and writes the results back as raw files.
 *
 *   round IN_DIR OUT_DIR
 *
 * IN_DIR/meta.txt holds, whitespace-separated:
 *   V T dtype n_chains n_seg n_rows n_nodes max_steps ld alpha tau
 * and the other input files hold the arrays of ps_subtree_batch and ps_tree in
 * native byte order: logits.bin (n_rows x ld elements, bf16 bit patterns or
 * float32), tokens.bin (int32), chain_seg0.bin, seg_cut.bin, seg_src.bin,
 * chain_node0.bin, acc.bin, rej.bin, req.bin (int32), seg_row0.bin (int64),
 * u.bin (float64).  OUT_DIR receives lp0.bin, lq.bin, log_ratio.bin,
 * log_accept.bin (float64), state_seg.bin, end_node.bin, k_delta.bin, path.bin
 * (int32) and status.txt (the scoring and walk status words).
 *
 * Exit status: 0 on success, 1 for a bad input file, 2 for an error that
 * libps reports, 3 for a CUDA runtime error.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ps.h"

static const char *in_dir;
static const char *out_dir;

/* Reads exactly `bytes` bytes of IN_DIR/name into a new host buffer. */
static void *read_input(const char *name, size_t bytes) {
    char path[4096];
    FILE *f;
    void *buf;
    snprintf(path, sizeof path, "%s/%s", in_dir, name);
    f = fopen(path, "rb");
    if (!f) {
        fprintf(stderr, "cannot open %s\n", path);
        exit(1);
    }
    buf = malloc(bytes > 0 ? bytes : 1);
    if (!buf || fread(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "short read of %s\n", path);
        exit(1);
    }
    fclose(f);
    return buf;
}

static void write_output(const char *name, const void *buf, size_t bytes) {
    char path[4096];
    FILE *f;
    snprintf(path, sizeof path, "%s/%s", out_dir, name);
    f = fopen(path, "wb");
    if (!f || fwrite(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot write %s\n", path);
        exit(1);
    }
    fclose(f);
}

static void check_cuda(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        exit(3);
    }
}

/* A device copy of `bytes` host bytes (at least one byte is allocated). */
static void *device_copy(const void *host, size_t bytes) {
    void *d = NULL;
    check_cuda(cudaMalloc(&d, bytes > 0 ? bytes : 1), "cudaMalloc");
    if (bytes > 0) check_cuda(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice), "copy in");
    return d;
}

static void *device_zeros(size_t bytes) {
    void *d = NULL;
    check_cuda(cudaMalloc(&d, bytes > 0 ? bytes : 1), "cudaMalloc");
    check_cuda(cudaMemset(d, 0, bytes > 0 ? bytes : 1), "cudaMemset");
    return d;
}

/* Copies a device array back and writes it to OUT_DIR/name. */
static void save(const char *name, const void *dev, size_t bytes) {
    void *h = malloc(bytes > 0 ? bytes : 1);
    if (!h) exit(1);
    if (bytes > 0) check_cuda(cudaMemcpy(h, dev, bytes, cudaMemcpyDeviceToHost), "copy out");
    write_output(name, h, bytes);
    free(h);
}

int main(int argc, char **argv) {
    int V, T, dtype, n_chains, n_seg, n_nodes, max_steps;
    long long n_rows_ll, ld_ll;
    double alpha, tau;
    size_t esz, n_rows, ld, path_len;
    FILE *meta;
    char path[4096];
    ps_subtree_batch b;
    ps_tree t;
    ps_score_out o;
    ps_walk_out wo;
    size_t ws_bytes;
    void *ws = NULL;
    ps_status st;
    int32_t status[2];
    char text[64];

    if (argc != 3) {
        fprintf(stderr, "usage: %s IN_DIR OUT_DIR\n", argv[0]);
        return 1;
    }
    in_dir = argv[1];
    out_dir = argv[2];
    snprintf(path, sizeof path, "%s/meta.txt", in_dir);
    meta = fopen(path, "r");
    if (!meta || fscanf(meta, "%d %d %d %d %d %lld %d %d %lld %lf %lf", &V, &T, &dtype,
                        &n_chains, &n_seg, &n_rows_ll, &n_nodes, &max_steps, &ld_ll, &alpha,
                        &tau) != 11) {
        fprintf(stderr, "bad %s\n", path);
        return 1;
    }
    fclose(meta);
    if (n_rows_ll < 0 || ld_ll < 1 || n_chains < 1 || n_seg < 1 || n_nodes < 1 ||
        max_steps < 0) {
        fprintf(stderr, "bad sizes in %s\n", path);
        return 1;
    }
    n_rows = (size_t)n_rows_ll;
    ld = (size_t)ld_ll;
    esz = dtype == PS_BF16 ? 2 : 4;
    path_len = (size_t)n_chains * (size_t)(max_steps + 1);

    memset(&b, 0, sizeof b);
    b.V = V;
    b.T = T;
    b.dtype = dtype;
    b.n_chains = n_chains;
    b.n_seg = n_seg;
    b.flags = 0;
    b.n_rows = (int64_t)n_rows;
    b.ld = (int64_t)ld;
    b.n_logit_rows = (int64_t)n_rows;
    b.alpha = alpha;
    b.tau = tau;
    b.eps = 0.01;
    b.chain_seg0 = device_copy(read_input("chain_seg0.bin", (n_chains + 1) * 4), (n_chains + 1) * 4);
    b.seg_row0 = device_copy(read_input("seg_row0.bin", (n_seg + 1) * 8), (n_seg + 1) * 8);
    b.seg_cut = device_copy(read_input("seg_cut.bin", n_seg * 4), n_seg * 4);
    b.seg_src = device_copy(read_input("seg_src.bin", n_seg * 4), n_seg * 4);
    b.logits = device_copy(read_input("logits.bin", n_rows * ld * esz), n_rows * ld * esz);
    b.tokens = device_copy(read_input("tokens.bin", n_rows * 4), n_rows * 4);

    memset(&t, 0, sizeof t);
    t.n_chains = n_chains;
    t.n_nodes = n_nodes;
    t.n_seg = n_seg;
    t.max_steps = max_steps;
    t.chain_node0 = device_copy(read_input("chain_node0.bin", (n_chains + 1) * 4), (n_chains + 1) * 4);
    t.chain_seg0 = b.chain_seg0;
    t.acc = device_copy(read_input("acc.bin", n_nodes * 4), n_nodes * 4);
    t.rej = device_copy(read_input("rej.bin", n_nodes * 4), n_nodes * 4);
    t.req = device_copy(read_input("req.bin", n_nodes * 4), n_nodes * 4);
    t.u = device_copy(read_input("u.bin", n_seg * 8), n_seg * 8);

    memset(&o, 0, sizeof o);
    o.lp0 = device_zeros(n_rows * 8);
    o.lq = device_zeros(n_rows * 8);
    o.log_ratio = device_zeros(n_seg * 8);
    o.log_accept = device_zeros(n_seg * 8);
    o.status = device_zeros(4);
    memset(&wo, 0, sizeof wo);
    wo.state_seg = device_zeros(n_chains * 4);
    wo.end_node = device_zeros(n_chains * 4);
    wo.k_delta = device_zeros(n_chains * 4);
    wo.path = device_zeros(path_len * 4);
    wo.status = device_zeros(4);

    ws_bytes = ps_score_workspace_bytes(&b);
    check_cuda(cudaMalloc(&ws, ws_bytes), "cudaMalloc workspace");   /* 256-byte aligned */
    st = ps_score_walk_subtree(&b, &t, &o, &wo, ws, ws_bytes, NULL);
    if (st != PS_OK) {
        fprintf(stderr, "ps_score_walk_subtree: %s\n", ps_status_string(st));
        return 2;
    }
    check_cuda(cudaDeviceSynchronize(), "synchronize");

    save("lp0.bin", o.lp0, n_rows * 8);
    save("lq.bin", o.lq, n_rows * 8);
    save("log_ratio.bin", o.log_ratio, n_seg * 8);
    save("log_accept.bin", o.log_accept, n_seg * 8);
    save("state_seg.bin", wo.state_seg, n_chains * 4);
    save("end_node.bin", wo.end_node, n_chains * 4);
    save("k_delta.bin", wo.k_delta, n_chains * 4);
    save("path.bin", wo.path, path_len * 4);
    check_cuda(cudaMemcpy(&status[0], o.status, 4, cudaMemcpyDeviceToHost), "copy status");
    check_cuda(cudaMemcpy(&status[1], wo.status, 4, cudaMemcpyDeviceToHost), "copy status");
    snprintf(text, sizeof text, "%d %d\n", (int)status[0], (int)status[1]);
    write_output("status.txt", text, strlen(text));
    printf("%s\n", ps_version());
    return 0;
}
