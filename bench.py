"""Benchmark of the tensor-parallel sharded linear pipeline on one B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--tp TP]
                    [--impl reference]

Default workload: the LLaMA-7B-shaped SwiGLU MLP block (2048 tokens, H=4096,
I=11008, bf16), sharded tp=8 ways in one device's memory. One step is one
pass of the block's hot path: the column-parallel gate/up GEMM with the
SwiGLU epilogue (tp_column_linear), then the row-parallel down GEMM with the
shard sum folded into its accumulator (tp_row_linear). Prints one JSON line.

Other workloads (--workload): gqa (attention projections, 4096 tokens, 32/8
heads, hd 128, tp 16 by default), decode (70B-like MLP at T tokens, tp 8,
HBM-bound), stack (4 LLaMA-7B blocks + 32000-vocab head, 4096 tokens, tp 4).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream; L2 is flushed before every timed step, outside the
events: a 256 MB write, then a 256 MB read that evicts the dirty lines. N>1 (torchrun): every rank runs an independent
replica of the workload on its own GPU (no collective on the data path);
the step time is the max over ranks.

--impl reference: the CPU oracle (float64 numpy) timed on this host's cores
on a bounded sample of the same workload (token rows are independent).
"""
from __future__ import annotations

import argparse
import math
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sharded MLP/attn-proj TFLOP/s & tokens/s at 1 B300; % of BF16 peak or HBM roofline"
E2E_WARMUP = 40     # untimed end-to-end steps per warm-up chunk
E2E_WARMUP_S = 1.0  # seconds of untimed end-to-end steps before the timed ones
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# Workload definitions (sizes of the pages' LLaMA-7B / 70B-shaped blocks)
# ---------------------------------------------------------------------------
def workload_spec(name: str, tp: int | None, tokens: int | None):
    if name == "mlp":
        T, H, I = tokens or 2048, 4096, 11008
        tp = tp or 8
        flops = 6.0 * T * H * I
        return dict(name="llama7b_swiglu_mlp", T=T, H=H, I=I, tp=tp, flops=flops,
                    dominant="col_swiglu_gemm (gate/up + SwiGLU epilogue)",
                    dominant_flops=4.0 * T * H * I, bound="tensor")
    if name == "mlp_bwd":
        # backward of the same MLP: 6 GEMMs of 2*T*H*I each (dHs, dW2, and the
        # input and weight gradients of gate and up)
        T, H, I = tokens or 2048, 4096, 11008
        tp = tp or 8
        return dict(name="llama7b_swiglu_mlp_backward", T=T, H=H, I=I, tp=tp, flops=12.0 * T * H * I,
                    dominant="weight-gradient GEMM of the gate shards (dW1, both operands MN-major), "
                             "timed through tp_column_linear_backward, whose interface keeps each shard's "
                             "gradient in its own tile rows (inside tp_mlp_backward the same product runs "
                             "over all of I at once)",
                    dominant_flops=2.0 * T * H * I, bound="tensor",
                    sample_note="the first {r} of {T} tokens, a complete backward problem of its own "
                                "(weight gradients sum over tokens)")
    if name == "moe":
        # a Mixtral-shaped MoE FFN: 8 SwiGLU experts (H=4096, I=14336), top-2
        # synthetic routing, every expert split over tp=8 shards; the work
        # counts the routed tokens only (not the units' padding rows)
        T, H, I, E, k = tokens or 4096, 4096, 14336, 8, 2
        tp = tp or 8
        fl = 6.0 * T * k * H * I
        return dict(name="moe_8x_swiglu_top2_tp", T=T, H=H, I=I, E=E, k=k, tp=tp, flops=fl,
                    dominant="moe block (dispatch, grouped gate/up + SwiGLU, grouped down + shard sum, combine)",
                    dominant_flops=fl, bound="tensor",
                    sample_note="{r} of {T} tokens (tokens are independent)")
    if name == "lm_ce":
        # the vocabulary-parallel ends of a language model: embedding lookup,
        # column-parallel LM head, vocabulary-parallel cross-entropy with its
        # gradient (the LM head of the 7B stack: V = 32000, tp = 4)
        T, H, V = tokens or 4096, 4096, 32000
        tp = tp or 4
        return dict(name="vocab_embedding_lm_head_cross_entropy", T=T, H=H, V=V, tp=tp, flops=2.0 * T * H * V,
                    dominant="lm_head_col_gemm with loss statistics in its epilogue (logits [tp][T][V/tp])",
                    dominant_flops=2.0 * T * H * V,
                    bound="tensor",
                    sample_note="{r} of {T} tokens (losses of different tokens are independent)")
    if name == "gqa":
        T, H, hq, hkv, hd = tokens or 4096, 4096, 32, 8, 128
        tp = tp or 16
        flops = 2.0 * T * H * (hq + 2 * hkv) * hd + 2.0 * T * hq * hd * H
        return dict(name="gqa_attn_proj", T=T, H=H, hq=hq, hkv=hkv, hd=hd, tp=tp, flops=flops,
                    dominant="qkv_col_gemm (QKV by heads, replicas computed once)",
                    dominant_flops=2.0 * T * H * (hq + 2 * hkv) * hd, bound="tensor")
    if name == "gqa_attn":
        # the GQA projections with the causal attention core between them;
        # the core's algorithmic FLOPs count only the visible (t' <= t) scores
        T, H, hq, hkv, hd = tokens or 4096, 4096, 32, 8, 128
        tp = tp or 16
        core = 2.0 * 2.0 * hd * hq * T * (T + 1) / 2.0
        flops = 2.0 * T * H * (hq + 2 * hkv) * hd + core + 2.0 * T * hq * hd * H
        return dict(name="gqa_attn_block_causal", T=T, H=H, hq=hq, hkv=hkv, hd=hd, tp=tp, flops=flops,
                    dominant="attention_core (causal, every local head)", dominant_flops=core,
                    bound="tensor",
                    sample_note="the first {r} of {T} tokens, a complete causal problem of its own",
                    flops_of_rows=lambda r: (2.0 * r * H * (hq + 2 * hkv) * hd + 2.0 * 2.0 * hd * hq * r * (r + 1) / 2.0
                                             + 2.0 * r * hq * hd * H))
    if name == "decode":
        T, H, I = tokens or 1, 8192, 28672
        tp = tp or 8
        wbytes = 3.0 * H * I * 2
        abytes = (T * H * 2) * 2 + T * I * 2 * 2   # X in, Y out, Hs write + read
        return dict(name="decode_70b_swiglu_mlp", T=T, H=H, I=I, tp=tp, flops=6.0 * T * H * I,
                    bytes=wbytes + abytes, dominant="col_swiglu_gemm (weight streaming)",
                    dominant_bytes=2.0 * H * I * 2 + T * H * 2 + T * I * 2, bound="hbm")
    if name == "stack":
        T, H, I, hq, hkv, hd, V, L = tokens or 4096, 4096, 11008, 32, 8, 128, 32000, 4
        tp = tp or 4
        attn = 2.0 * T * H * (hq + 2 * hkv) * hd + 2.0 * T * hq * hd * H
        mlp = 6.0 * T * H * I
        flops = L * (attn + mlp) + 2.0 * T * H * V
        return dict(name="llama7b_stack4_lmhead", T=T, H=H, I=I, hq=hq, hkv=hkv, hd=hd, V=V, L=L, tp=tp,
                    flops=flops, dominant="col_swiglu_gemm (one block's gate/up + SwiGLU)",
                    dominant_flops=4.0 * T * H * I,
                    bound="tensor")
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------
# CPU oracle leg (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return int(max(n)) if n else (os.cpu_count() or 1)
    except Exception:
        return os.cpu_count() or 1


class OracleLeg:
    """The CPU oracle on a sample of the workload's token rows (rows are
    independent in every workload here, so a row sample is the same
    computation on fewer tokens)."""

    def __init__(self, spec):
        import synth_inputs as S
        from oracle import tp_oracle as O
        self.spec, name, tp, T = spec, spec["name"], spec["tp"], spec["T"]
        if name.startswith("moe_"):
            H, I, E, k = spec["H"], spec["I"], spec["E"], spec["k"]
            X = S.normal(70, (T, H))[:min(T, 64)].astype(np.float64)
            ex = [{kk: v.astype(np.float64) for kk, v in e.items()} for e in S.moe_experts(E, H, I)]
            ids, w = S.moe_routing(71, T, E, k)
            self.fn = lambda r: O.moe_tp(X[:r], ex, ids[:r], w[:r].astype(np.float64), tp)
        elif name.startswith("vocab_embedding_lm_head"):
            H, V = spec["H"], spec["V"]
            d = S.vocab_lm(min(T, 256), H, V)
            E, W = d["E"].astype(np.float64), d["W_lm"].astype(np.float64)
            ids, labels = d["ids"], d["labels"]
            self.fn = lambda r: O.vocab_parallel_cross_entropy(
                O.column_parallel(O.vocab_embedding(ids[:r], E, tp), W, tp), labels[:r])
            X = ids
        elif name.startswith("llama7b_swiglu_mlp_backward"):
            H, I = spec["H"], spec["I"]
            d = S.mlp_backward(min(T, 512), H, I)
            Wg, Wu, Wd = (d[k].astype(np.float64) for k in ("Wg", "Wu", "Wd"))
            X, dY = d["X"].astype(np.float64), d["dY"].astype(np.float64)
            # the first r tokens: a complete backward problem of its own
            self.fn = lambda r: O.mlp_backward(X[:r], Wg, Wd, tp, dY[:r], "swiglu", W_up=Wu)
        elif name.startswith("llama7b_swiglu") or name.startswith("decode"):
            H, I = spec["H"], spec["I"]
            d = (S.swiglu_mlp(min(T, 512), H, I) if name.startswith("llama7b")
                 else S.decode_mlp(min(T, 512), H, I))
            Wg, Wu, Wd = (d[k].astype(np.float64) for k in ("Wg", "Wu", "Wd"))
            X = d["X"].astype(np.float64)
            self.fn = lambda r: O.mlp_block(X[:r], Wg, Wd, tp, "swiglu", W_up=Wu)
        elif name.startswith("gqa"):
            H, hq, hkv, hd = spec["H"], spec["hq"], spec["hkv"], spec["hd"]
            d = S.gqa_proj(min(T, 512), H, hq, hkv, hd)
            A = {k: d[k].astype(np.float64) for k in d}
            X = A["X"]
            core = "causal" if name.startswith("gqa_attn_block") else None
            # the first r tokens: a complete causal problem of its own
            self.fn = lambda r: O.attn_proj(X[:r], A["Wq"], A["Wk"], A["Wv"], A["Wo"], hq, hkv, hd, tp,
                                            attention=core)
        else:
            d = S.stack(min(T, 128))
            Ls = [{k: v.astype(np.float64) for k, v in L.items()} for L in d["layers"]]
            Wlm = d["W_lm"].astype(np.float64)
            X = d["X"].astype(np.float64)
            self.fn = lambda r: O.stack_forward(X[:r], Ls, Wlm, tp, spec["hq"], spec["hkv"], spec["hd"])
        self.avail = X.shape[0]

    def calibrate(self, target_s):
        rows = 1
        while True:
            t0 = time.perf_counter()
            self.fn(rows)
            dt = time.perf_counter() - t0
            if dt >= 0.5 * target_s or rows >= self.avail:
                break
            rows = min(self.avail, max(rows * 2, int(rows * 0.8 * target_s / max(dt, 1e-3))))
        return rows

    def value(self, rows, elapsed):
        sp = self.spec
        if sp["bound"] == "hbm":  # algorithmic bytes of a rows-token problem, bf16 storage
            per_tok = (sp["bytes"] - 3.0 * sp["H"] * sp["I"] * 2) / sp["T"]
            return (3.0 * sp["H"] * sp["I"] * 2 + rows * per_tok) / elapsed / 1e9
        if "flops_of_rows" in sp:
            return sp["flops_of_rows"](rows) / elapsed / 1e12
        return sp["flops"] / sp["T"] * rows / elapsed / 1e12

    def timed(self, rows):
        t0 = time.perf_counter()
        self.fn(rows)
        return time.perf_counter() - t0


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------
class ClockSampler:
    """Samples SM clocks and clock-event (throttle) reasons while the timed
    region runs, with `nvidia-smi --query-gpu ... -lms 20` in a child process
    (the same fields as the profiling recipe's clocks line). Only samples
    whose timestamps fall inside the marked timed window are summarised."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,power.draw")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, local_index: int, period_ms: int = 20):
        self.rows, self.error, self.window = [], None, None
        self.proc, self._t = None, None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.target = vis.split(",")[local_index] if vis else str(local_index)
        self.period_ms = period_ms

    def _reader(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.perf_counter(), parts))

    def start(self):
        import subprocess
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._reader, daemon=True)
            self._t.start()
            time.sleep(0.5)  # nvidia-smi's first sample arrives a few hundred ms after start
        except Exception as e:  # no nvidia-smi: the line then says so
            self.error = repr(e)

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            time.sleep(2 * self.period_ms / 1000.0)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=5)

    def summary(self):
        rows = self.rows
        if self.window:
            t0, t1 = self.window
            inside = [r for r in rows if t0 <= r[0] <= t1 + 0.03]
            rows = inside
        mhz, mx, reasons, watts = [], None, set(), []
        for _, p in rows:
            try:
                mhz.append(float(p[0]))
                mx = float(p[1])
                watts.append(float(p[6]))
            except ValueError:
                continue
            for nm, v in zip(self.NAMES, p[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        out = {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
               "reasons": sorted(reasons), "samples": len(mhz),
               "power_w_median": statistics.median(watts) if watts else None}
        if self.error:
            out["sampler_error"] = self.error
        return out


def rank_info():
    """(rank, world size, local rank) from the launcher's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest of each rank's value (the job's time is its slowest rank's)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha(files=None) -> str:
    """sha256 prefix over the named csrc files (all of them by default), so
    that a change to one kernel's sources leaves the others' records valid."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_transformer_linear_tma_b300", "csrc")
    for f in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str, T: int):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources of that kernel (the files its record lists) and at
    this token count (null otherwise)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{workload}:{kernel}")
    if not e or e.get("source_sha") != kernel_source_sha(e.get("source_files")) or e.get("T") != T:
        return None
    return e.get("dram_bytes_per_launch")


def setup_workload(spec, torch, tpl):
    """Generate seeded inputs on the host, upload, shard. Returns a dict with
    the step callables and the buffers they use."""
    import synth_inputs as S
    B = torch.bfloat16
    up = lambda a: torch.from_numpy(a).to("cuda").to(B)
    name, tp, T = spec["name"], spec["tp"], spec["T"]
    st = {}
    if name.startswith("moe_"):
        H, I, E, k = spec["H"], spec["I"], spec["E"], spec["k"]
        ex = S.moe_experts(E, H, I)
        Wg = tpl.tp_shard_experts([up(e["W1"]) for e in ex], tp, "col")
        Wu = tpl.tp_shard_experts([up(e["W_up"]) for e in ex], tp, "col")
        Wd = tpl.tp_shard_experts([up(e["W2"]) for e in ex], tp, "row")
        del ex
        X = up(S.normal(70, (T, H)))
        ids_h, w_h = S.moe_routing(71, T, E, k)
        ids = torch.from_numpy(ids_h).to("cuda")
        wts = torch.from_numpy(w_h).to("cuda")
        Y = torch.empty((T, H), dtype=B, device="cuda")
        ws = torch.empty(tpl.tp_moe_workspace_bytes(T, H, I, k, E, tp), dtype=torch.uint8, device="cuda")

        def api_call(Xin, Yout):  # dispatch (3), grouped gate/up, grouped down, combine: 6 launches
            tpl.tp_moe_block(Xin, ids, wts, Wg, Wu, Wd, E, workspace=ws, out=Yout)
        st.update(parts=[lambda: api_call(X, Y)], X=X, Y=Y, api=api_call, launches_per_step=6,
                  keep=[Wg, Wu, Wd, ids, wts, ws])
    elif name.startswith("vocab_embedding_lm_head"):
        H, V = spec["H"], spec["V"]
        d = S.vocab_lm(T, H, V)
        E = up(d["E"])
        Slm = tpl.tp_shard_weights(up(d["W_lm"]), tp, "col")
        ids = torch.from_numpy(d["ids"]).to("cuda")
        labels = torch.from_numpy(d["labels"]).to("cuda")
        del d
        X0 = torch.empty((T, H), dtype=B, device="cuda")
        logits = torch.empty((tp, T, V // tp), dtype=B, device="cuda")
        loss = torch.empty(T, dtype=torch.float32, device="cuda")
        mean = torch.empty(1, dtype=torch.float32, device="cuda")
        ws = torch.empty(max(tpl.lib.tp_lm_head_ce_workspace_bytes(T, Slm.ref()), 256), dtype=torch.uint8,
                         device="cuda")

        def p_embed(ids_in=ids):
            tpl.tp_vocab_embedding(ids_in, E, tp, out=X0)

        def p_head_ce(mean_out=mean):
            # LM head with the loss statistics in its epilogue, the per-token
            # combine, the mean and the gradient of the mean loss (in place)
            tpl.tp_lm_head_cross_entropy(X0, Slm, labels, logits=logits, dlogits=logits, workspace=ws, loss=loss,
                                         mean_loss=mean_out)

        def p_dominant():  # the LM head GEMM with its statistics epilogue (+ the small combine)
            tpl.tp_lm_head_cross_entropy(X0, Slm, labels, logits=logits, workspace=ws, loss=loss,
                                         want_mean=False)

        def api_call(ids_in, mean_out):  # ids in, mean loss out: 1 + 4 launches
            p_embed(ids_in)
            p_head_ce(mean_out)
        st.update(parts=[p_embed, p_head_ce], X=ids, Y=mean, api=api_call, launches_per_step=5,
                  keep=[E, Slm, labels, X0, logits, loss, ws], dominant_part=p_dominant)
    elif name.startswith("llama7b_swiglu_mlp_backward"):
        H, I = spec["H"], spec["I"]
        d = S.mlp_backward(T, H, I)
        Sg = tpl.tp_shard_weights(up(d["Wg"]), tp, "col")
        Su = tpl.tp_shard_weights(up(d["Wu"]), tp, "col")
        Sd = tpl.tp_shard_weights(up(d["Wd"]), tp, "row")
        X, dY = up(d["X"]), up(d["dY"])
        del d
        # the forward's saved values, computed once outside the timed region
        G = tpl.tp_column_linear(X, Sg, act="none")
        U = tpl.tp_column_linear(X, Su, act="none")
        Hs = tpl.tp_column_linear(X, Sg, W_up=Su, act="swiglu")
        Is = I // tp
        grads = {"dX": torch.empty((T, H), dtype=B, device="cuda"),
                 "dW1": torch.empty((tp, Is, H), dtype=B, device="cuda"),
                 "dW_up": torch.empty((tp, Is, H), dtype=B, device="cuda"),
                 "dW2": torch.empty((tp, H, Is), dtype=B, device="cuda")}
        ws = torch.empty(tpl.tp_mlp_backward_workspace_bytes(T, H, I, tp, "swiglu", B), dtype=torch.uint8,
                         device="cuda")

        def api_call(dYin, dXout):  # the whole backward: 5 GEMM launches and the activation gradient
            tpl.tp_mlp_backward(X, Sg, Sd, G, Hs, dYin, W_up=Su, U=U, act="swiglu", workspace=ws,
                                out=dict(grads, dX=dXout))

        def part_a():  # the gate shards' weight-gradient GEMM alone
            tpl.tp_column_linear_backward(X, Sg, G, want_dX=False, want_dW=True)
        st.update(parts=[lambda: api_call(dY, grads["dX"])], X=dY, Y=grads["dX"], api=api_call,
                  launches_per_step=6, keep=[Sg, Su, Sd, X, G, U, Hs, grads, ws], dominant_part=part_a)
    elif name.startswith("llama7b_swiglu") or name.startswith("decode"):
        H, I = spec["H"], spec["I"]
        d = S.swiglu_mlp(T, H, I) if name.startswith("llama7b") else S.decode_mlp(T, H, I)
        Sg = tpl.tp_shard_weights(up(d["Wg"]), tp, "col")
        Su = tpl.tp_shard_weights(up(d["Wu"]), tp, "col")
        Sd = tpl.tp_shard_weights(up(d["Wd"]), tp, "row")
        X = up(d["X"])
        del d
        Hs = torch.empty((tp, T, I // tp), dtype=B, device="cuda")
        Y = torch.empty((T, H), dtype=B, device="cuda")
        ws = torch.empty(max(tpl.tp_mlp_workspace_bytes(T, H, I, tp, B), 256), dtype=torch.uint8, device="cuda")
        gws = torch.empty(max(tpl.tp_gemm_workspace_bytes(T, Sg), tpl.tp_gemm_workspace_bytes(T, Sd), 256),
                          dtype=torch.uint8, device="cuda")

        def api_call(Xin, Yout):  # column GEMM + SwiGLU, then row GEMM + sum: two launches
            tpl.tp_mlp_block(Xin, Sg, Sd, W_up=Su, act="swiglu", workspace=ws, out=Yout)

        def part_a():  # the column launch of tp_mlp_block, timed alone
            tpl.tp_column_linear(X, Sg, W_up=Su, act="swiglu", out=Hs, workspace=gws)
        st.update(parts=[lambda: api_call(X, Y)], X=X, Y=Y, api=api_call, launches_per_step=2,
                  keep=[Sg, Su, Sd, Hs, ws, gws], dominant_part=part_a)
    elif name.startswith("gqa_attn_block"):
        H, hq, hkv, hd = spec["H"], spec["hq"], spec["hkv"], spec["hd"]
        d = S.gqa_proj(T, H, hq, hkv, hd)
        Sqkv = tpl.tp_shard_qkv(up(d["Wq"]), up(d["Wk"]), up(d["Wv"]), hq, hkv, hd, tp)
        So = tpl.tp_shard_weights(up(d["Wo"]), tp, "row")
        X = up(d["X"])
        del d
        qkv = torch.empty((tp, T, Sqkv.shard_width), dtype=B, device="cuda")
        ctx = torch.empty((tp, T, hq // tp * hd), dtype=B, device="cuda")
        Y = torch.empty((T, H), dtype=B, device="cuda")
        ws = torch.empty(max(tpl.tp_attn_workspace_bytes(T, hq, hkv, hd, tp, B), 256), dtype=torch.uint8,
                         device="cuda")

        def api_call(Xin, Yout):  # QKV GEMM, attention core, O GEMM + sum: three launches
            tpl.tp_attn_block(Xin, Sqkv, So, attention="causal", qkv_out=qkv, workspace=ws, out=Yout)

        def part_a():  # the attention core alone, on the step's qkv
            tpl.tp_attention(qkv, hq, hkv, hd, causal=True, out=ctx)
        st.update(parts=[lambda: api_call(X, Y)], X=X, Y=Y, api=api_call, launches_per_step=3,
                  keep=[Sqkv, So, qkv, ctx, ws], dominant_part=part_a)
    elif name.startswith("gqa"):
        H, hq, hkv, hd = spec["H"], spec["hq"], spec["hkv"], spec["hd"]
        d = S.gqa_proj(T, H, hq, hkv, hd)
        Sqkv = tpl.tp_shard_qkv(up(d["Wq"]), up(d["Wk"]), up(d["Wv"]), hq, hkv, hd, tp)
        So = tpl.tp_shard_weights(up(d["Wo"]), tp, "row")
        X = up(d["X"])
        del d
        Ns = Sqkv.shard_width
        qkv = torch.empty((tp, T, Ns), dtype=B, device="cuda")
        ctx = torch.empty((tp, T, hq // tp * hd), dtype=B, device="cuda")
        Y = torch.empty((T, H), dtype=B, device="cuda")
        ws = torch.empty(max(tpl.tp_attn_workspace_bytes(T, hq, hkv, hd, tp, B), 256), dtype=torch.uint8,
                         device="cuda")

        gws = torch.empty(max(tpl.tp_gemm_workspace_bytes(T, Sqkv), 256), dtype=torch.uint8, device="cuda")

        def part_a():  # the QKV launch of tp_attn_proj, timed alone
            tpl.tp_column_linear(X, Sqkv, out=qkv, workspace=gws)

        def api_call(Xin, Yout):
            # QKV by heads (its epilogue also writes the single-key context),
            # then O + shard sum: two launches
            tpl.tp_attn_proj(Xin, Sqkv, So, qkv_out=qkv, workspace=ws, out=Yout)
        st.update(parts=[lambda: api_call(X, Y)], X=X, Y=Y, api=api_call, launches_per_step=2,
                  keep=[Sqkv, So, qkv, ctx, ws, gws], dominant_part=part_a)
    else:
        H, I, hq, hkv, hd, V, L = (spec[k] for k in ("H", "I", "hq", "hkv", "hd", "V", "L"))
        d = S.stack(T, H, I, hq, hkv, hd, V, L)
        layers = []
        for Lw in d["layers"]:
            layers.append(dict(
                qkv=tpl.tp_shard_qkv(up(Lw["Wq"]), up(Lw["Wk"]), up(Lw["Wv"]), hq, hkv, hd, tp),
                o=tpl.tp_shard_weights(up(Lw["Wo"]), tp, "row"),
                g=tpl.tp_shard_weights(up(Lw["Wg"]), tp, "col"),
                u=tpl.tp_shard_weights(up(Lw["Wu"]), tp, "col"),
                d=tpl.tp_shard_weights(up(Lw["Wd"]), tp, "row")))
        lm = tpl.tp_shard_weights(up(d["W_lm"]), tp, "col")
        # the residual stream is fp32 (its values start as the bf16 inputs);
        # norms write bf16 GEMM inputs; the LM head writes bf16 logits
        X = torch.from_numpy(d["X"]).to("cuda")
        del d
        x1 = torch.empty_like(X)
        h = torch.empty(X.shape, dtype=B, device="cuda")
        logits = torch.empty((T, V), dtype=B, device="cuda")
        wa = torch.empty(max(tpl.tp_attn_workspace_bytes(T, hq, hkv, hd, tp, B), 256), dtype=torch.uint8, device="cuda")
        wm = torch.empty(max(tpl.tp_mlp_workspace_bytes(T, H, I, tp, B), 256), dtype=torch.uint8, device="cuda")

        def forward(Xin, out):
            x = Xin
            for Lw in layers:
                tpl.tp_rmsnorm(x, out=h)
                tpl.tp_attn_proj(h, Lw["qkv"], Lw["o"], residual=x, workspace=wa, out=x1)
                tpl.tp_rmsnorm(x1, out=h)
                tpl.tp_mlp_block(h, Lw["g"], Lw["d"], W_up=Lw["u"], residual=x1, act="swiglu",
                                 workspace=wm, out=x1)  # in-place residual add
                x = x1
            tpl.tp_rmsnorm(x, out=h)
            tpl.tp_column_linear(h, lm, concat=True, out=out)
        Hs1 = torch.empty((tp, T, I // tp), dtype=B, device="cuda")
        wg = torch.empty(max(tpl.tp_gemm_workspace_bytes(T, layers[0]["g"]), 256), dtype=torch.uint8, device="cuda")

        def part_a():  # one block's gate/up column launch, timed alone
            tpl.tp_column_linear(h, layers[0]["g"], W_up=layers[0]["u"], act="swiglu", out=Hs1, workspace=wg)
        st.update(parts=[lambda: forward(X, logits)], X=X, Y=logits, api=forward,
                  launches_per_step=L * 6 + 2, keep=[layers, lm, x1, h, wa, wm, Hs1, wg], dominant_part=part_a)
    return st


def run_gpu(args, spec):
    import torch
    import tensor_transformer_linear_tma_b300 as tpl

    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    st = setup_workload(spec, torch, tpl)
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_out = torch.empty((), dtype=torch.float32, device="cuda")

    def flush_l2(k):
        # Cold L2 before each timed step: write a buffer larger than L2, then
        # read another one so that the dirty lines are written back now rather
        # than inside the next timed kernel.
        flush_w.fill_(float(k))
        torch.amax(flush_r, dim=0, out=flush_out)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    clk = ClockSampler(local)
    if rank == 0:
        clk.start()
    for w in range(args.warmup):
        flush_l2(w)  # (its kernels load before the timed region too)
        for p in st["parts"]:
            p()
        if "dominant_part" in st:
            st["dominant_part"]()
    if tpl.tp_get_error() != 0:
        raise SystemExit("device error during warm-up")

    # The device-timed steps replay a CUDA graph of each part, captured after
    # warm-up (the same launches with the same arguments), so that host-side
    # time between the start event and the first launch cannot enter the
    # measurement when the host is slower than the GPU. The end-to-end leg
    # below calls the public API directly.
    launch_mode = "direct calls"
    if not args.no_graph:
        try:
            graphs = {}
            torch.cuda.synchronize()
            for key, fn in [(i, p) for i, p in enumerate(st["parts"])] + (
                    [("dominant", st["dominant_part"])] if "dominant_part" in st else []):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    fn()
                graphs[key] = g
            torch.cuda.synchronize()
            if tpl.tp_get_error() != 0:
                raise RuntimeError("device error during capture")
            st["parts"] = [graphs[i].replay for i in range(len(st["parts"]))]
            if "dominant" in graphs:
                st["dominant_part"] = graphs["dominant"].replay
            st["graphs"] = graphs
            for p in st["parts"]:  # one replay of each before timing
                p()
            torch.cuda.synchronize()
            launch_mode = "one CUDA graph replay per part (captured after warm-up)"
        except Exception as e:  # capture unavailable: time the direct calls
            launch_mode = f"direct calls (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()

    nparts = len(st["parts"])
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nparts + 1)] for _ in range(args.steps)]
    barrier()
    t_begin = time.perf_counter()
    for k in range(args.steps):
        flush_l2(k)
        e = evs[k]
        e[0].record(stream)
        for i, p in enumerate(st["parts"]):
            p()
            e[i + 1].record(stream)
    barrier()
    t_end = time.perf_counter()
    t_wall = t_end - t_begin
    clk.mark(t_begin, t_end)
    clk.stop()
    status = tpl.tp_get_error()
    if status != 0:
        raise SystemExit(f"device error in timed region: {tpl.tp_status_string(status)}")
    step_ms = [evs[k][0].elapsed_time(evs[k][nparts]) for k in range(args.steps)]
    part_ms = [[evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps)] for i in range(nparts)]
    ms = max_over_ranks(float(np.mean(step_ms)), dist, "cuda")

    # dominant kernel: its own launch duration over the timed steps
    if "dominant_part" in st:
        dom_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for k in range(args.steps):
            flush_l2(k)
            dom_ev[k][0].record(stream)
            st["dominant_part"]()
            dom_ev[k][1].record(stream)
        torch.cuda.synchronize()
        dom_ms = float(np.mean([a.elapsed_time(b) for a, b in dom_ev]))
    elif spec["name"].startswith("llama7b_stack"):
        dom_ms = None
    else:
        dom_ms = float(np.mean(part_ms[0]))

    # End to end through the public call with host buffers. Every step copies
    # its own input from pinned host memory and reads its own result back;
    # three streams (upload, compute, download) over double-buffered device
    # buffers let step k+1's upload and step k-1's download run under step
    # k's compute. The time is the wall time of all K steps (CUDA events on
    # the download stream), divided by K.
    nb = 2  # device and host buffers are rings of two (host copies are never read during timing)
    Xh = [torch.empty(st["X"].shape, dtype=st["X"].dtype, pin_memory=True) for _ in range(nb)]
    for x in Xh:
        x.copy_(st["X"].cpu())
    Yh = [torch.empty(st["Y"].shape, dtype=st["Y"].dtype, pin_memory=True) for _ in range(nb)]
    Xd = [torch.empty_like(st["X"]) for _ in range(nb)]
    Yd = [torch.empty_like(st["Y"]) for _ in range(nb)]
    s_up, s_cmp, s_dn = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    n_ev = max(args.steps, E2E_WARMUP, args.warmup)
    e_up = [torch.cuda.Event() for _ in range(n_ev)]
    e_cmp = [torch.cuda.Event() for _ in range(n_ev)]
    e_dn = [torch.cuda.Event() for _ in range(n_ev)]

    def e2e_run(n):
        for k in range(n):
            i = k % nb
            with torch.cuda.stream(s_up):
                if k >= nb:
                    s_up.wait_event(e_cmp[k - nb])   # compute of step k-nb has read Xd[i]
                Xd[i].copy_(Xh[i], non_blocking=True)
                e_up[k].record(s_up)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(e_up[k])
                if k >= nb:
                    s_cmp.wait_event(e_dn[k - nb])   # download of step k-nb has read Yd[i]
                st["api"](Xd[i], Yd[i])
                e_cmp[k].record(s_cmp)
            with torch.cuda.stream(s_dn):
                s_dn.wait_event(e_cmp[k])
                Yh[i].copy_(Yd[i], non_blocking=True)
                e_dn[k].record(s_dn)

    # Untimed warm-up of the pipeline, by wall time. On this host the first
    # few hundred milliseconds of transfers run well under the link's rate
    # (the MLP pipeline measured 0.80 ms a step over its first 400 steps,
    # 0.47 ms over the next 400, with the host enqueueing 70-140 us a step),
    # so the pipeline runs for E2E_WARMUP_S before the clock starts.
    t_warm = time.perf_counter()
    n_warm = 0
    while n_warm < args.warmup or time.perf_counter() - t_warm < E2E_WARMUP_S:
        e2e_run(E2E_WARMUP)
        torch.cuda.synchronize()
        n_warm += E2E_WARMUP
    barrier()
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0e.record(s_up)
    s_cmp.wait_event(t0e)
    s_dn.wait_event(t0e)
    e2e_run(args.steps)
    t1e.record(s_dn)
    barrier()
    e2e_ms = max_over_ranks(t0e.elapsed_time(t1e) / args.steps, dist, "cuda")

    peaks, peak_src = load_peaks()
    out = None
    if rank == 0:
        bound = spec["bound"]
        if bound == "hbm":
            value = spec["bytes"] * world / (ms * 1e-3) / 1e9
            unit = "GB/s"
            e2e_value = spec["bytes"] * world / (e2e_ms * 1e-3) / 1e9
            peak = peaks["hbm_gbs"]
            achieved = spec["dominant_bytes"] / (dom_ms * 1e-3) / 1e9 if dom_ms else None
        else:
            value = spec["flops"] * world / (ms * 1e-3) / 1e12
            unit = "TFLOP/s"
            e2e_value = spec["flops"] * world / (e2e_ms * 1e-3) / 1e12
            # The burst peak, unless the power cap actually held the clock down
            # during the timed region (median SM clock under 90% of its max):
            # then the sustained peak, measured under the same condition.
            clocks_now = clk.summary()
            mhz, mx = clocks_now.get("sm_mhz"), clocks_now.get("sm_max_mhz")
            capped = bool(mhz and mx and mhz < 0.9 * mx)
            peak = peaks["bf16_tflops_sustained" if capped else "bf16_tflops"]
            achieved = spec["dominant_flops"] / (dom_ms * 1e-3) / 1e12 if dom_ms else None
        clocks = clk.summary()
        cfg = {k: v for k, v in spec.items() if k in ("T", "H", "I", "hq", "hkv", "hd", "V", "L", "E", "k", "tp")}
        cfg.update(workload=spec["name"], tokens_per_step=spec["T"], launches=launch_mode,
                   l2="flushed before every timed step (256 MB write, then 256 MB read to evict it)",
                   layout=f"tp={spec['tp']} shards in one device's memory")
        out = {
            "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded normal inputs, random-init weights of the named shapes)",
            "config": cfg,
            "tokens_per_s": round(spec["T"] * world / (ms * 1e-3), 1),
            "tflops": round(spec["flops"] * world / (ms * 1e-3) / 1e12, 3),
            "frac_of_peak": round(value / peak, 4),
            "frac_of_burst_peak": round(value / peaks.get("bf16_tflops", peak), 4) if bound != "hbm" else None,
            "roofline": {
                "kernel": spec["dominant"], "bound": bound,
                "achieved": round(achieved, 3) if achieved else None,
                "peak": peak,
                "peak_source": f"{peak_src} " + ("(hbm_gbs)" if bound == "hbm" else
                                                 "(bf16_tflops_sustained: the power cap held the median SM clock under 90% of max)"
                                                 if peak == peaks.get("bf16_tflops_sustained") else
                                                 "(bf16_tflops burst)"),
                "unit": unit, "frac": round(achieved / peak, 4) if achieved else None,
                "traffic": ncu_traffic(spec["dominant"], spec["name"], spec["T"]),
                "kernel_ms": round(dom_ms, 5) if dom_ms else None,
            },
            "part_ms": [round(float(np.mean(p)), 5) for p in part_ms],
            # first and last tenth of the timed steps: the drift shows the power cap settling in
            "step_ms_first_last_tenth": [round(float(np.mean(step_ms[:max(1, len(step_ms) // 10)])), 5),
                                         round(float(np.mean(step_ms[-max(1, len(step_ms) // 10):])), 5)],
            "e2e": {"value": round(e2e_value, 3), "unit": unit,
                    "h2d_bytes_per_step": int(st["X"].numel() * st["X"].element_size()),
                    "d2h_bytes_per_step": int(st["Y"].numel() * st["Y"].element_size()),
                    "ms_per_step": round(e2e_ms, 5),
                    "copies": "pinned host buffers; upload/compute/download pipelined on 3 streams",
                    "l2": "not flushed between e2e steps; each step touches more than the 126 MB L2"},
            "gpu_launches": st["launches_per_step"] * args.steps,
            "clocks": clocks,
            "wall_s_timed": round(t_wall, 4),
        }
    if dist is not None:
        dist.destroy_process_group()
    return out


def cpu_baseline_obj(spec, unit, target_s):
    leg = OracleLeg(spec)
    rows = leg.calibrate(target_s)
    # the sample is capped at the rows prepared for the oracle: repeat the pass
    # until about target_s of CPU work has been timed
    first = leg.timed(rows)
    passes = max(1, min(200, int(math.ceil(0.9 * target_s / max(first, 1e-3)))))
    total = first + sum(leg.timed(rows) for _ in range(passes - 1))
    what = spec.get("sample_note", "{r} of {T} token rows (rows are independent)").format(r=rows, T=spec["T"])
    return {"value": round(leg.value(rows, total / passes), 6), "unit": unit, "cores": _blas_threads(),
            "kind": "oracle",
            "sample": f"{what}, {passes} pass{'es' if passes > 1 else ''}, float64 numpy oracle, {total:.2f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mlp",
                    choices=["mlp", "mlp_bwd", "gqa", "gqa_attn", "decode", "stack", "lm_ce", "moe"])
    ap.add_argument("--tp", type=int, default=None)
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time direct calls instead of graph replays")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    spec = workload_spec(args.workload, args.tp, args.tokens)
    rank = rank_info()[0]
    unit = "GB/s" if spec["bound"] == "hbm" else "TFLOP/s"

    if args.impl == "reference":
        if rank != 0:
            return
        leg = OracleLeg(spec)
        per = max(1.0, min(args.cpu_seconds, 90.0 / max(args.steps, 1)))
        rows = leg.calibrate(per)
        for _ in range(min(args.warmup, 1)):
            leg.timed(rows)
        t0 = time.perf_counter()
        times = [leg.timed(rows) for _ in range(args.steps)]
        wall = time.perf_counter() - t0
        v = leg.value(rows, float(np.mean(times)))
        what = spec.get("sample_note", "{r} of {T} token rows (rows are independent)").format(r=rows, T=spec["T"])
        sample = f"{what} per step, float64 numpy oracle, {np.mean(times):.3f} s per step"
        line = {"metric": METRIC, "value": round(v, 6), "unit": unit, "n_gpus": 1, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(wall * 1e3 / args.steps, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference",
                "config": {"workload": spec["name"], "tp": spec["tp"], "T": spec["T"]},
                "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": _blas_threads(),
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    # the CPU baseline runs first, before any CUDA context exists
    cpu = None
    if rank == 0 and args.gpus == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_obj(spec, unit, args.cpu_seconds)
    out = run_gpu(args, spec)
    if out is not None:
        out["cpu_baseline"] = cpu
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
