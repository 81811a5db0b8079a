// Internal state shared by the planner, the runtime glue and the kernels' host
// launchers.  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include <vector_types.h>

#include "spinf.h"

namespace spinf {

constexpr int kTile = 128;  // rows of a Q tile and of a KV tile

// Device copies of one pass's descriptors, in one allocation.
struct PassDevice {
    void* block = nullptr;
    bool owned = true;             // false: caller-owned memory (spinf_plan_upload_to)
    int32_t* end = nullptr;        // [T_pad]
    int32_t* pos = nullptr;        // [T_pad]
    int32_t* tile_ptr = nullptr;   // [n_qtiles + 1]
    int32_t* tile_kv = nullptr;    // [n_sched]
    int32_t* tile_len = nullptr;   // [n_sched]
    int32_t* slot_row = nullptr;   // [M]
    int32_t* gather_m = nullptr;   // [G]
    int32_t* gather_tok = nullptr; // [G]
    int32_t* row_gptr = nullptr;   // [M + 1] gathers of each scoring row ...
    int32_t* row_glist = nullptr;  // [G]     ... sorted by token id, then gather index
    int32_t* qt_work = nullptr;    // [n_qtiles][4] attention work order {qt, s0, n, 0}, most KV tiles first
    int32_t* row_runs = nullptr;   // [T_pad][8] root path of each row as <= 4 runs [lo, hi) (lo0 -1: more)
    int32_t* row_x = nullptr;      // [M] searched-slot index of each scoring row, or -1
    int32_t* x_m = nullptr;        // [X] scoring row of each searched slot
    int32_t* x_set = nullptr;      // [X] allowed-token set of each searched slot (-1: every token)
};

// The KV-tile schedule of one pass for a sliding window W: the W = 0 schedule without
// the tiles in which no row of the Q tile sees any key within W (built on first use).
struct WindowSchedule {
    int32_t window = 0;      // 0: no window
    int32_t key_tile = 128;  // keys per KV tile: 128, or 64 (the halves of the 128-key tiles)
    int32_t q_rows = 128;    // rows per Q tile: 128, or 64 (the halves of the planner's Q tiles)
    std::vector<int32_t> tile_ptr, tile_kv, tile_len, qt_work;
    void* block = nullptr;   // device copies of qt_work, tile_kv, tile_len (plan-owned)
    bool in_pass_block = false;   // the copies sit in the pass's descriptor block (the 64-key schedule)
    int32_t *d_qt_work = nullptr, *d_tile_kv = nullptr, *d_tile_len = nullptr;
    std::vector<unsigned char> staging;
};

// cos and sin of the rotary angles of one pass for one (d_head, theta): [d / 2][max pos + 1]
// (built on first use, plan-owned device copy).
struct RopeTable {
    int32_t d = 0;
    int32_t stride = 0;   // max pos + 1
    float theta = 0.f;
    std::vector<float2> host;
    float2* dev = nullptr;
};

struct Pass {
    int32_t T = 0, T_pad = 0;
    std::vector<int32_t> tok, parent, pos, end, anchor;
    std::vector<int32_t> tile_ptr, tile_kv, tile_len, qt_work, row_runs;
    std::vector<int32_t> slot_row, gather_m, gather_tok;
    std::vector<int32_t> row_gptr, row_glist;
    std::vector<int32_t> x_m, x_set, row_x;   // searched slots: scoring row, token set; per scoring row its slot or -1
    std::vector<int32_t> unit_start, unit_source;
    PassDevice dev;
    std::vector<unsigned char> staging;   // host source of the descriptor upload, kept until the plan is freed
    std::vector<std::unique_ptr<WindowSchedule>> windows;
    std::vector<std::unique_ptr<RopeTable>> ropes;
};

// Where the option tokens of one laid-out question sit in its pass's gather list.
struct QuestionSite {
    int32_t pass = -1;
    int32_t g0 = 0;          // first gather entry
    int32_t opt0 = 0;        // first entry in Plan::opt_len
    int32_t n_options = 0;
    int32_t x = -1;          // searched slot: index in its pass's x_m / x_set
};

}  // namespace spinf

struct spinf_plan {
    std::vector<spinf::Pass> passes;
    std::vector<int32_t> opt_len;                // token count of every option, question by question
    std::vector<spinf::QuestionSite> user_q;     // every user question, input by input
    std::vector<int32_t> user_q_floor;           // floor index per user question, or -1
    std::vector<spinf::QuestionSite> floor_q;    // every floor question
    int64_t n_options_total = 0;
    int64_t n_extract = 0;                       // searched slots among the user questions
    int32_t extract_k = 8;
    std::mutex cache_mu;                         // guards the lazily built per-pass caches (windows, rotary tables)
    int32_t* d_err = nullptr;                    // device error word (allocated at first upload)
    bool err_owned = true;                       // false: inside a caller-owned descriptor buffer
    int device = -1;
};

namespace spinf {
spinf_status fail(spinf_status s, const std::string& msg);
spinf_status ok();
// The pass's schedule for window W > 0, built on first use and kept by the plan.
WindowSchedule& window_schedule(Pass& P, int32_t window);
// The schedule for window W >= 0 in KV tiles of `key_tile` keys (128 or 64) and Q tiles of
// `q_rows` rows (128 or 64), built on first use.
WindowSchedule& tile_schedule(Pass& P, int32_t window, int32_t key_tile, int32_t q_rows = kTile);
}  // namespace spinf
