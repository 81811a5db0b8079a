/* A C caller of the library with no Python in between: plan one request, read its
 * pass, and collect results from hand-set token log-probabilities (host calls only).
 * Prints: passes T M G questions options p0 p1 residual floor_p0 floor_p1 floor_residual;
 * then, for a request with a searched slot: n_extract k X tok0 tok1 lp0 lp1 residual-is-NaN and
 * the two scored questions' residuals. */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "spinf.h"

int main(void) {
    const int32_t content[] = {1, 2, 3, 4}, tmpl[] = {5, 6}, o1[] = {7}, o2[] = {8, 9};
    const spinf_tokens opts[2] = {{o1, 1}, {o2, 2}};
    spinf_question q;
    memset(&q, 0, sizeof q);
    q.tmpl.ids = tmpl;
    q.tmpl.n = 2;
    q.options = opts;
    q.n_options = 2;
    q.kind = SPINF_Q_SCORED;
    q.token_set = -1;
    spinf_input in;
    memset(&in, 0, sizeof in);
    in.content.ids = content;
    in.content.n = 4;
    in.questions = &q;
    in.n_questions = 1;
    spinf_plan_opts o;
    spinf_plan_opts_default(&o);
    o.vocab = 100;
    spinf_plan* plan = NULL;
    if (spinf_pack_plan(&in, 1, &o, &plan) != SPINF_OK) {
        fprintf(stderr, "plan: %s\n", spinf_last_error());
        return 1;
    }
    spinf_pass_info info;
    int64_t nq = 0, no = 0;
    if (spinf_plan_pass_info(plan, 0, &info) != SPINF_OK || spinf_plan_counts(plan, &nq, &no) != SPINF_OK) return 2;
    /* gather order: the user question's tokens 7 | 8 9, then its floor's */
    const float tlp[6] = {logf(0.5f), logf(0.25f), logf(0.5f), logf(0.5f), logf(0.5f), logf(0.5f)};
    const float* per_pass[1] = {tlp};
    double lp[2], p[2], flp[2], fp[2], res[1], fres[1];
    spinf_result r = {lp, p, flp, fp, res, fres};
    if (spinf_collect(plan, per_pass, &r) != SPINF_OK) return 3;
    printf("%d %d %d %d %lld %lld %.9f %.9f %.9f %.9f %.9f %.9f\n", spinf_plan_num_passes(plan), info.T, info.M,
           info.G, (long long)nq, (long long)no, p[0], p[1], res[0], fp[0], fp[1], fres[0]);
    spinf_plan_free(plan);

    /* a searched slot ({*}: any token) between two scored questions, extract_k 2 */
    const int32_t t2[] = {10, 11};
    spinf_question qs[3];
    qs[0] = q;
    memset(&qs[1], 0, sizeof qs[1]);
    qs[1].tmpl.ids = t2;
    qs[1].tmpl.n = 2;
    qs[1].kind = SPINF_Q_SEARCHED;
    qs[1].token_set = -1;
    qs[2] = q;
    in.questions = qs;
    in.n_questions = 3;
    o.extract_k = 2;
    if (spinf_pack_plan(&in, 1, &o, &plan) != SPINF_OK) {
        fprintf(stderr, "plan: %s\n", spinf_last_error());
        return 4;
    }
    int64_t n_x = 0;
    int32_t k = 0;
    if (spinf_plan_extract_counts(plan, &n_x, &k) != SPINF_OK || spinf_plan_pass_info(plan, 0, &info) != SPINF_OK)
        return 5;
    const int32_t top_tok[2] = {42, 17};
    const float top_lp[2] = {-0.5f, -1.5f};
    const int32_t* tt[1] = {top_tok};
    const float* tl[1] = {top_lp};
    int32_t tok_out[2];
    double lp_out[2];
    if (spinf_collect_extract(plan, tt, tl, tok_out, lp_out) != SPINF_OK) return 6;
    /* token lps of the scored questions (two of them, one floor they share) */
    float tlp2[9];
    for (int i = 0; i < 9; ++i) tlp2[i] = tlp[i % 3];
    const float* pp2[1] = {tlp2};
    double lp2[4], p2[4], flp2[4], fp2[4], res2[3], fres2[3];
    spinf_result r2 = {lp2, p2, flp2, fp2, res2, fres2};
    if (spinf_collect(plan, pp2, &r2) != SPINF_OK) return 7;
    printf("%lld %d %d %d %d %.3f %.3f %d %.9f %.9f\n", (long long)n_x, k, info.X, tok_out[0], tok_out[1], lp_out[0],
           lp_out[1], isnan(res2[1]) ? 1 : 0, res2[0], res2[2]);
    spinf_plan_free(plan);
    return 0;
}
