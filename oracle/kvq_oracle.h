/*
 * CPU oracle for the quantized KV cache -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline leg may load or call this code.  It shares nothing with the CUDA
 * library (no headers, helpers, tables or constants) and never calls it.
 *
 * Everything here is plain scalar C: fp32 quantization exactly as the formula
 * states it (IEEE round-to-nearest-even, no contraction), fp64 attention over
 * the dequantized cache.  One head (one batch entry, one KV head) at a time.
 *
 * Sources (page title, section):
 *   [KIVI]    "大模型量化技术原理：KIVI、IntactKV、KVQuant" (juejin), KIVI / 背景,
 *             为什么键和值缓存应该沿着不同的维度进行量化, 工作原理.
 *   [KVQ2]    same page, KVQuant / 技术原理 二 (keys quantized before the rotary
 *             position embedding, the embedding applied after dequantization).
 *   [KVQ4]    same page, KVQuant / 技术原理 四 (per-vector dense-and-sparse:
 *             each vector's outliers kept apart in fp16, the rest quantized
 *             over a narrower range; per-token thresholds computed online).
 *   [KVQ5]    same page, KVQuant / 技术原理 五、Attention Sink 感知量化.
 *   [IKV]     same page, IntactKV / KV Cache量化 (fp16 part concatenated with
 *             the dequantized cache at inference time).
 *   [HF]      pgsm.cn KV-cache quantization how-to, §2.1 量化基础概念,
 *             §3.1 残差缓存设计, §3.2 内存节省计算示例.
 *   [INNERQ]  "【论文】InnerQ：硬件感知免调优KV缓存量化用于大语言模型" (euno.news),
 *             关键贡献, 方法论 1-4.
 *
 * Parity unpinned: orc_choose_symmetric's threshold.  The InnerQ page asks
 * for the symmetric mode when a group is centred at zero and gives no
 * threshold; the rule here (midpoint within half an asymmetric step of zero)
 * is a choice.  Its implementation is pinned by worked boundary cases, the
 * rule itself by nothing on the pages.  The other readings where the pages
 * are silent (the value queue's pop, fp16 metadata rounding, the outlier
 * count and tie rule, the rotary pairing) are each pinned against their
 * stated definition.
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_KIVI 0
#define ORC_INNERQ 1

/* Per-head cache state.  Every array is owned by the caller. */
typedef struct orc_head {
  int32_t d;          /* head_dim */
  int32_t bits;       /* 2, 4 or 8 */
  int32_t scheme;     /* ORC_KIVI or ORC_INNERQ */
  int32_t k_group;    /* KIVI: tokens per key group G; InnerQ: channels per key group */
  int32_t v_group;    /* channels per value group */
  int32_t residual;   /* KIVI: residual length R; InnerQ: recent window W */
  int32_t n_sink;     /* InnerQ: fp16 sink tokens S */
  int32_t k_normalize;/* InnerQ: 1 = one-shot per-channel key normalization */
  int64_t cap;        /* token capacity of the quantized region */
  int64_t n_quant;    /* tokens held quantized */
  int64_t n_resid;    /* KIVI: fp16 residual tokens; InnerQ: fp16 window tokens */
  int64_t n_sink_used;/* InnerQ: sink tokens held */
  int64_t n_flush;    /* KIVI: residual flushes so far */
  uint8_t *k_u, *v_u;         /* [cap][d], one code per byte */
  float *k_scale, *k_zero;    /* KIVI [cap/G][d];  InnerQ [cap][d/k_group] */
  float *v_scale, *v_zero;    /* [cap][d/v_group] */
  uint8_t *k_sym, *v_sym;     /* InnerQ [cap][d/group]: 1 = symmetric group */
  uint16_t *k_res, *v_res;    /* [residual][d] fp16, oldest first */
  uint16_t *k_sink, *v_sink;  /* [n_sink][d] fp16 */
  float *k_norm;              /* InnerQ with k_normalize: [d] per-channel key factors */
  int32_t v_queue;            /* KIVI: 1 = values leave fp16 one at a time (a queue) */
  int64_t n_vquant;           /* KIVI with v_queue: values held quantized */
  int32_t meta_f16;           /* 1 = scales and zeros stored in fp16 */
  int32_t outliers;           /* KIVI: fp16 outliers kept per token and tensor (0 = none) */
  uint16_t *k_oidx, *v_oidx;  /* [cap][outliers] channels of each token's outliers, ascending */
  uint16_t *k_oval, *v_oval;  /* [cap][outliers] their fp16 values */
} orc_head;

int orc_rounding_is_nearest(void);
float orc_half_to_float(uint16_t h);
uint16_t orc_float_to_half(float f);

void orc_quant_asym(const float *x, int n, int bits, float *scale, float *zero,
                    uint8_t *u, int64_t ustride);
void orc_quant_sym(const float *x, int n, int bits, float *scale, float *zero,
                   uint8_t *u, int64_t ustride);
int orc_choose_symmetric(float mn, float mx, int bits);
void orc_quant_asym_f16(const float *x, int n, int bits, float *scale, float *zero,
                        uint8_t *u, int64_t ustride);
void orc_quant_sym_f16(const float *x, int n, int bits, float *scale, float *zero,
                       uint8_t *u, int64_t ustride);

int orc_prefill(orc_head *s, const uint16_t *K, const uint16_t *V, int64_t T);
int orc_append(orc_head *s, const uint16_t *k, const uint16_t *v);
int orc_attend(const orc_head *s, const uint16_t *q, double tau, double *out);
int orc_attend_rope(const orc_head *s, const uint16_t *q, double tau, double base,
                    int64_t pos0, double *out);

void orc_select_outliers(const uint16_t *row, int d, int k, uint16_t *idx);
void orc_pack(const uint8_t *u, int64_t n_rows, int d, int bits, uint8_t *out);
void orc_pack_modes(const uint8_t *sym, int64_t n, uint32_t *out);

#ifdef __cplusplus
}
#endif
#endif
