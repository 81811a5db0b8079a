/* A C caller of the library with no Python in between: plan one request, read its
 * pass, and collect results from hand-set token log-probabilities (host calls only).
 * Prints: passes T M G questions options p0 p1 residual floor_p0 floor_p1 floor_residual. */
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
    return 0;
}
