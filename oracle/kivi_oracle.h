/*
 * kivi_oracle.h -- declarations of the CPU oracle (test infrastructure only;
 * see kivi_oracle.c).  All fp16 values travel as their IEEE binary16 bit
 * patterns in uint16_t.
 */
#ifndef KIVI_ORACLE_H
#define KIVI_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ko_cache ko_cache;

float ko_f16_to_f32(uint16_t h);
uint16_t ko_f32_to_f16(float f);

/* Quantize n values x[i*stride] with B = bits; writes the fp16 scale and
 * zero and the codes codes[i*code_stride]. */
void ko_quantize_group(const float *x, int n, int stride, int bits,
                       uint16_t *s_out, uint16_t *z_out,
                       uint8_t *codes, int code_stride);
float ko_dequant(uint8_t code, uint16_t s16, uint16_t z16);

/* 0 ok, 1 invalid argument, 2 out of memory, 3 capacity exceeded */
int ko_create(int b, int h, int d, int kbits, int vbits, int G, int R, int cap,
              ko_cache **out);
void ko_destroy(ko_cache *o);
int ko_prefill(ko_cache *o, const uint16_t *K, const uint16_t *V,
               const int *t, int t_stride);
int ko_append(ko_cache *o, const uint16_t *k, const uint16_t *v);
int ko_decode(const ko_cache *o, const uint16_t *q, int hq, float *out);
int ko_decode_subset(const ko_cache *o, const uint16_t *q, int hq, float *out,
                     const int *pairs, int npairs);
int ko_decode_probs(const ko_cache *o, const uint16_t *q, int hq, float *out,
                    float *probs, long long ld, const int *pairs, int npairs);
int ko_set_threads(int n);
int ko_prefill_attn(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int *t, int b, int hq,
                    int h, int ts, int d, const int *rows, int nrows, double *out);
void ko_f32_to_f16_n(const float *x, uint16_t *y, size_t n);
void ko_f16_to_f32_n(const uint16_t *x, float *y, size_t n);
void ko_lengths(const ko_cache *o, int *T, int *Tqk, int *Tqv);
void ko_dequant_kv(const ko_cache *o, int i, int j, float *Khat, float *Vhat);
void ko_state(const ko_cache *o, uint8_t *kcode, uint16_t *ks, uint16_t *kz,
              uint8_t *vcode, uint16_t *vs, uint16_t *vz, uint16_t *kf, uint16_t *vf);
int ko_capacity(const ko_cache *o);
int ko_capacity_stride(const ko_cache *o);

int ko_export_supported(const ko_cache *o);
void ko_export_sizes(const ko_cache *o, size_t *n_kc, size_t *n_ksz, size_t *n_vc,
                     size_t *n_vsz, size_t *n_kf, size_t *n_vf);
int ko_export(const ko_cache *o, uint32_t *Kc, uint16_t *Ksz, uint32_t *Vc,
              uint16_t *Vsz, uint16_t *Kf, uint16_t *Vf);

#ifdef __cplusplus
}
#endif
#endif
