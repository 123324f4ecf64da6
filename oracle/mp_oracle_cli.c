/*
 * mp_oracle_cli.c — command-line front end of the CPU oracle (TEST
 * INFRASTRUCTURE ONLY, like the oracle itself): runs the oracle on raw
 * little-endian binary files so that results can be produced or checked
 * without Python.
 *
 *   mp_oracle_cli step N TABLE PARAMS GRADS MASTER|- M V LR BETA1 BETA2 EPS WD CLIP T SEED
 *       One optimizer step over N parameters, in place on the files: the
 *       gradient norm and clip scale (oracle_grad_norm), then
 *       oracle_adamw_step. TABLE is a text file of "offset size decay" lines
 *       tiling [0, N); PARAMS and GRADS hold bf16 patterns (uint16), MASTER,
 *       M and V fp32 ("-" for MASTER selects the no-master variant). Prints
 *       "norm <value> scale <value> status <code>".
 *   mp_oracle_cli sr N IN OUT GLOBAL_OFFSET SEED
 *       OUT (bf16 patterns) = stochastic rounding of IN (fp32).
 *   mp_oracle_cli sr16 N IN OUT GLOBAL_OFFSET SEED
 *       OUT (fp16 patterns) = stochastic rounding of IN (fp32) to fp16.
 *   mp_oracle_cli noise FIRST N SEED
 *       Prints the N rounding draws from global index FIRST, one hex word per line.
 * Exit status 0 on success, 1 on a usage or I/O error, 2 if the step refused.
 */
#include <inttypes.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mp_oracle.h"

static void* read_file(const char* path, size_t bytes)
{
    FILE* f = fopen(path, "rb");
    if (!f)
        return NULL;
    void* buf = malloc(bytes ? bytes : 1);
    const size_t got = buf ? fread(buf, 1, bytes, f) : 0;
    fclose(f);
    if (!buf || got != bytes) {
        free(buf);
        return NULL;
    }
    return buf;
}

static int write_file(const char* path, const void* buf, size_t bytes)
{
    FILE* f = fopen(path, "wb");
    if (!f)
        return 0;
    const size_t put = fwrite(buf, 1, bytes, f);
    return fclose(f) == 0 && put == bytes;
}

static oracle_tensor* read_table(const char* path, uint64_t n, int32_t* count)
{
    FILE* f = fopen(path, "r");
    if (!f)
        return NULL;
    int32_t cap = 64, k = 0;
    oracle_tensor* t = malloc(sizeof *t * (size_t)cap);
    uint64_t off, size, covered = 0;
    int decay;
    while (t && fscanf(f, "%" SCNu64 " %" SCNu64 " %d", &off, &size, &decay) == 3) {
        if (k == cap) {
            cap *= 2;
            oracle_tensor* grown = realloc(t, sizeof *t * (size_t)cap);
            if (!grown) {
                free(t);
                t = NULL;
                break;
            }
            t = grown;
        }
        if (off != covered || (decay != 0 && decay != 1)) {
            free(t);
            t = NULL;
            break;
        }
        t[k].offset = off;
        t[k].size = size;
        t[k].decay = decay;
        t[k].pad = 0;
        covered += size;
        ++k;
    }
    fclose(f);
    if (t && covered != n) {
        free(t);
        t = NULL;
    }
    *count = k;
    return t;
}

static int cmd_step(int argc, char** argv)
{
    if (argc != 17)
        return 1;
    const uint64_t n = strtoull(argv[2], NULL, 10);
    int32_t nt = 0;
    oracle_tensor* table = read_table(argv[3], n, &nt);
    uint16_t* params = read_file(argv[4], n * 2);
    uint16_t* grads = read_file(argv[5], n * 2);
    const int with_master = strcmp(argv[6], "-") != 0;
    float* master = with_master ? read_file(argv[6], n * 4) : NULL;
    float* m = read_file(argv[7], n * 4);
    float* v = read_file(argv[8], n * 4);
    if (!table || !params || !grads || (with_master && !master) || !m || !v)
        return 1;
    const float lr = strtof(argv[9], NULL), beta1 = strtof(argv[10], NULL), beta2 = strtof(argv[11], NULL);
    const float eps = strtof(argv[12], NULL), wd = strtof(argv[13], NULL), clip = strtof(argv[14], NULL);
    const int32_t t = (int32_t)strtol(argv[15], NULL, 10);
    const uint32_t seed = (uint32_t)strtoul(argv[16], NULL, 10);
    double sumsq;
    float norm, scale;
    oracle_grad_norm(grads, n, clip, &sumsq, &norm, &scale);
    const int st = oracle_adamw_step(params, grads, master, m, v, 0, n, table, nt, lr, beta1, beta2, eps, wd,
                                     scale, t, seed);
    printf("norm %.9g scale %.9g status %d\n", norm, scale, st);
    int ok = st == 0 && write_file(argv[4], params, n * 2) && write_file(argv[7], m, n * 4) &&
             write_file(argv[8], v, n * 4) && (!with_master || write_file(argv[6], master, n * 4));
    free(table); free(params); free(grads); free(master); free(m); free(v);
    return st != 0 ? 2 : (ok ? 0 : 1);
}

static int cmd_sr(int argc, char** argv, int to_fp16)
{
    if (argc != 7)
        return 1;
    const uint64_t n = strtoull(argv[2], NULL, 10);
    float* in = read_file(argv[3], n * 4);
    uint16_t* out = malloc(n > 0 ? n * 2 : 1);
    if (!in || !out)
        return 1;
    const uint64_t goff = strtoull(argv[5], NULL, 10);
    const uint32_t seed = (uint32_t)strtoul(argv[6], NULL, 10);
    if (to_fp16)
        oracle_stochastic_round_fp16(out, in, goff, n, seed);
    else
        oracle_stochastic_round(out, in, goff, n, seed);
    const int ok = write_file(argv[4], out, n * 2);
    free(in); free(out);
    return ok ? 0 : 1;
}

static int cmd_noise(int argc, char** argv)
{
    if (argc != 5)
        return 1;
    const uint64_t first = strtoull(argv[2], NULL, 10), n = strtoull(argv[3], NULL, 10);
    const uint32_t seed = (uint32_t)strtoul(argv[4], NULL, 10);
    for (uint64_t i = 0; i < n; ++i)
        printf("%08" PRIx32 "\n", oracle_noise_u32(first + i, seed));
    return 0;
}

int main(int argc, char** argv)
{
    int rc = 1;
    if (argc >= 2 && strcmp(argv[1], "step") == 0)
        rc = cmd_step(argc, argv);
    else if (argc >= 2 && strcmp(argv[1], "sr") == 0)
        rc = cmd_sr(argc, argv, 0);
    else if (argc >= 2 && strcmp(argv[1], "sr16") == 0)
        rc = cmd_sr(argc, argv, 1);
    else if (argc >= 2 && strcmp(argv[1], "noise") == 0)
        rc = cmd_noise(argc, argv);
    if (rc == 1)
        fprintf(stderr, "usage: see the header of mp_oracle_cli.c (bad arguments or files)\n");
    return rc;
}
