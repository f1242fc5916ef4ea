/*
 * CPU oracle for the split-residency routed MoE layer -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg call
 * this code.  The CUDA library never links, includes or calls it, and this
 * file shares no code, table or constant generator with it.
 *
 * Sources (pages of the write-up series on cold expert residency):
 *  - "vLLM: Pin Hot Experts", Results: the layer runs the routed MXFP4 expert
 *    FFN once per residency bank without finalize, then one finalize
 *    accumulates each token's k bf16 expert rows in fp32 with fma in the
 *    original k order and casts once; so the split is bit-identical to the
 *    unsplit layer.  Section "Making it follow the traffic" and E4/E4b: true
 *    swaps (hot row to staging, cold row into the hot slot, staging into the
 *    cold slot, then the two-element row-map write).
 *  - "We Built the Counter", section 2: one masked relaxed atomic add per
 *    routed pick into a [layers x experts] int32 table; only steps of at most
 *    256 tokens are counted; stale-proof swaps decided against a CPU copy of
 *    the hot/cold lists.  Section 9: policy defaults (read every 64 steps,
 *    500-step half-life, <=2 swaps per layer per read, 1.5x hysteresis,
 *    minimum average 8, <=8 swaps per step).
 *  - MXFP4 itself (e2m1 elements, e8m0 scale per 32 elements) follows the OCP
 *    Microscaling Formats (MX) v1.0 specification, which the pages name only
 *    as "MXFP4" with "ue8m0 block scales".
 *
 * Precision: dot products accumulate in double; g, u, h and the expert output
 * row are then held in fp32 as the plain "fp32 expert FFN"; the expert row is
 * rounded once to bf16 (the "bf16 expert rows" the finalize reads).  The
 * finalize uses C99 fmaf, which is correctly rounded.  Build with
 * -ffp-contract=off so no other fused operation appears.
 *
 * Parity pins: every function here is pinned by tests (hand-decoded values,
 * closed forms, brute force, invariants); see tests/test_oracle_pins.py.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- MXFP4 element and scale decode (OCP MX v1.0, FP4 E2M1 / E8M0) ---- */
double orc_e2m1_value(unsigned code);          /* code in 0..15 */
double orc_e8m0_value(unsigned byte);          /* NaN for 0xFF */
/* Dequantise rows x K of packed e2m1 (K/2 bytes per row, low nibble = even
 * K index) with one e8m0 scale per 32 K-elements into out[rows][K]. */
void orc_dequant(const uint8_t *q, const uint8_t *s, int64_t rows, int64_t K, double *out);

/* ---- bf16 helpers ---- */
float orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);             /* round to nearest even */

/* ---- router (the step that produces the logits) ----
 * "vLLM: Pin Hot Experts", Where the experts live today: the router scores
 * every expert for every token.  logits[t][e] = fp32(bias[e] + sum_h
 * x[t][h] * w_router[e][h]) with bf16 x and w_router widened exactly, the sum
 * taken in double and rounded to fp32 once.  bias may be NULL (zero). */
void orc_router_logits(const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int E, int H,
                       float *logits);

/* ---- routing: top-k over fp32 logits, softmax over the k picks ----
 * ids[t][j]: the j-th largest logit of token t (ties: lower expert id first);
 * w[t][j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k picks, in fp32,
 * summed in j order.  The pages assume finite logits; a NaN logit is read
 * as -infinity for both the ranking and the weights (reading: a score that
 * is not a number ranks below every score, so k valid ids always come out). */
void orc_route(const float *logits, int T, int E, int k, int32_t *ids, float *w);

/* ---- residency: row map and split ----
 * row_map[e] >= 0: expert e lives in hot-bank row row_map[e];
 * row_map[e] <  0: expert e lives in cold-bank row -1 - row_map[e].
 * Initial placement: hot rows are assigned to the hot experts in increasing
 * expert id, cold rows likewise. */
void orc_initial_rowmap(const uint8_t *is_hot, int E, int32_t *row_map, int *n_hot, int *n_cold);

/* Per-bank pick lists (bank 0 = hot, 1 = cold).  For each bank: the active
 * local rows in increasing order (n_act of them), the offset of each active
 * row's picks (n_act + 1 entries), and the picks themselves as slot indices
 * t*k + j, ordered by (local row, slot).  Arrays are sized T*k (+1). */
typedef struct {
    int32_t n_picks[2];
    int32_t n_act[2];
    int32_t *act_row[2];   /* [T*k]   */
    int32_t *act_off[2];   /* [T*k+1] */
    int32_t *picks[2];     /* [T*k]   */
} orc_split_t;
void orc_split(const int32_t *row_map, int E, const int32_t *ids, int T, int k, orc_split_t *out);

/* Usage counter: counts[e] += 1 per pick when count_on and T <= count_tmax. */
void orc_count(int32_t *counts, int E, const int32_t *ids, int T, int k, int count_on, int count_tmax);

/* ---- expert FFN ----
 * One expert, n tokens: g = W_gate x, u = W_up x (double dot products, held
 * in fp32), h = silu(g) * u with silu(z) = z / (1 + exp(-z)) in fp32,
 * y = W2 h (double dot product, fp32, then bf16).  x rows and y rows are bf16
 * bit patterns [n][H].  Weights are the logical layout of one expert. */
void orc_expert_ffn(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                    const uint8_t *w2_s, int H, int I, const uint16_t *x, int n, uint16_t *y);

/* ---- MXFP8 activations (the opt-in one-piece prefill format) ----
 * The pages do not state the activation format of the routed MXFP4 kernel
 * ("vLLM: Pin Hot Experts", Where the experts live today).  This reading is
 * the OCP MX v1.0 MXFP8 format: blocks of 32 consecutive elements share a
 * power of two 2^e, elements are FP8 E4M3 (round to nearest even, saturating
 * at +-448).  e is the smallest integer with amax * 2^-e <= 448, so no element
 * saturates, held to the e8m0 range [-127, 127].
 * orc_e4m3_rne: the E4M3 value nearest v (ties to even), saturated.
 * orc_mx8_block_exponent: e for a block whose largest |value| is amax.
 * orc_mx8_quantize: the MXFP8 reading of v (n % 32 == 0), as doubles.
 * orc_expert_ffn_mx8: orc_expert_ffn with the token rows (qx != 0) and the
 * gate/up output h (qh != 0) read as MXFP8 before the GEMM that consumes
 * them; qx = qh = 0 is orc_expert_ffn exactly. */
double orc_e4m3_rne(double v);
int orc_mx8_block_exponent(double amax);
void orc_mx8_quantize(const double *v, int64_t n, double *out);
void orc_expert_ffn_mx8(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                        const uint8_t *w2_s, int H, int I, const uint16_t *x, int n, uint16_t *y,
                        int qx, int qh);

/* ---- finalize ----
 * out[t][c] = bf16( fma-chain over j = 0..k-1 of w[t][j] * Y[t][j][c] ),
 * accumulator fp32 starting at +0, one cast at the end. */
void orc_finalize(const uint16_t *Y, const float *w, int T, int k, int H, uint16_t *out);

/* ---- whole layer-step ----
 * Weights: all E experts of the layer in the logical layout, stacked.
 * Computes ids, w, Y (the unfinalized expert rows [T][k][H]) and out [T][H];
 * counts (may be NULL) is updated per orc_count. */
void orc_layer_step(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                    const uint8_t *w2_s, int E, int k, int H, int I,
                    const float *logits, const uint16_t *x, int T,
                    int32_t *ids, float *w, uint16_t *Y, uint16_t *out,
                    int32_t *counts, int count_on, int count_tmax);

/* Expert rows for a subset of slots only (sampled parity at full size):
 * for each of the n_slots slot indices s = t*k + j, compute Y[s] (H bf16) from
 * the given ids.  Y_out is [n_slots][H]. */
void orc_rows_for_slots(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                        const uint8_t *w2_s, int H, int I, int k, const int32_t *ids,
                        const uint16_t *x, const int32_t *slots, int n_slots,
                        uint16_t *Y_out);
/* The same with mx8 != 0: x and h read as MXFP8 (orc_expert_ffn_mx8). */
void orc_rows_for_slots_fmt(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                            const uint8_t *w2_s, int H, int I, int k, const int32_t *ids,
                            const uint16_t *x, const int32_t *slots, int n_slots,
                            uint16_t *Y_out, int mx8);

/* ---- swaps (true swaps with stale check) ----
 * For each pair i in order: promote[i] must currently be cold and demote[i]
 * hot (checked against row_map, which is the CPU copy of the placement);
 * otherwise applied[i] = 0 and nothing changes.  An applied pair exchanges
 * the two experts' rows: promote takes demote's hot row, demote takes
 * promote's cold row.  Returns the number applied. */
int orc_swap(int32_t *row_map, int E, int n, const int32_t *promote, const int32_t *demote,
             int32_t *applied);

/* ---- restore to a saved placement ----
 * "We Built the Counter", section 2: an operator may ask for the start-up
 * placement back, and a round trip of swaps back to the start-up hot set
 * leaves the output unchanged.  Reading: a restore brings back the
 * saved HOT SET; which row of a bank an expert occupies changes no output.
 * Pairs: the experts cold in row_map and hot in target (ascending id) are
 * promoted, each against the next expert hot in row_map and cold in target
 * (ascending id); at most max_pairs pairs.  Returns the pair count, or -1
 * when the two maps have different hot counts. */
int orc_plan_restore(const int32_t *row_map, const int32_t *target, int E, int max_pairs,
                     int32_t *promote, int32_t *demote);

/* ---- adaptive policy (host side, between steps) ----
 * State per layer: the last counts read, an exponentially decaying sum of the
 * per-read pick deltas and the matching decaying sum of weights.  At a read:
 *   delta_e = counts_e - last_e  (uint32 difference),
 *   d = 0.5^(read_every / half_life),
 *   acc_e = d * acc_e + delta_e,  wsum = d * wsum + 1,
 *   avg_e = acc_e / wsum          (decaying average, picks per read).
 * Candidates: cold experts with avg >= min_avg, by avg descending; hot
 * experts by avg ascending (ties: lower expert id first).  Pair the i-th of
 * each while i < max_pairs and avg_cold > hysteresis * avg_hot.
 * Returns the number of pairs written to promote/demote. */
typedef struct {
    int E;
    uint32_t *last;
    double *acc;
    double wsum;
} orc_policy_t;
void orc_policy_init(orc_policy_t *p, int E, uint32_t *last, double *acc, const int32_t *counts);
int orc_policy_read(orc_policy_t *p, const int32_t *counts, const int32_t *row_map,
                    double read_every, double half_life, double hysteresis, double min_avg,
                    int max_pairs, int32_t *promote, int32_t *demote);

/* ---- byte model ---- */
int64_t orc_expert_bytes(int H, int I);

int orc_num_threads(void);
void orc_set_num_threads(int n);   /* threads of the OpenMP loops (n > 0) */

#ifdef __cplusplus
}
#endif
#endif
