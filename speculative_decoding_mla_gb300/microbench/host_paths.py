"""Where the host's time goes in one verify call (one GPU).

For a workload (default long_185k) this prints, as one JSON object:
  copies          pinned-memory copies of the host-buffer call's sizes, each timed alone to the
                  synchronisation: the kv_indices and q host-to-device, out device-to-host, and an
                  empty synchronisation;
  host_call_us    verify_attn_mla_host (q, indices and results crossing) timed to its return;
  device_call_us  the same call on device buffers (verify_attn_mla), timed to the synchronisation;
  submit          the device-buffer call's host time alone (the stream held by a sleep kernel, so
                  the whole call is queued before the GPU reaches it), the device time of the
                  queued call between two events, and the call's wall time from an idle GPU.
Medians over the repetitions.

    python -m speculative_decoding_mla_gb300.microbench.host_paths long_185k contiguous_1k
"""
import json
import sys
import time

import numpy as np


def _median_wall(fn, n, torch):
    ts = []
    for _ in range(n):
        torch.cuda.synchronize()
        a = time.perf_counter()
        fn()
        torch.cuda.synchronize()
        ts.append(time.perf_counter() - a)
    return float(np.median(ts) * 1e6)


def measure(name, reps=30):
    import torch
    from speculative_decoding_mla_gb300 import build
    build.build()  # the binding loads the library when it is imported
    from speculative_decoding_mla_gb300 import binding, device, synth
    case = synth.workload(name)
    dc = device.to_device(case)
    T, H = case.q.shape[0], case.num_heads
    res = {"workload": name}

    # the host-buffer call's transfers, each alone
    q_h = torch.from_numpy(case.q.view(np.int16)).pin_memory()
    kvi_h = torch.from_numpy(case.kv_indices).pin_memory()
    out_h = torch.empty((T, H, 512), dtype=torch.int16).pin_memory()
    lse_h = torch.empty((T, H), dtype=torch.float32).pin_memory()
    q_d, kvi_d, out_d = (torch.empty_like(x, device="cuda") for x in (q_h, kvi_h, out_h))
    res["copies"] = {
        "h2d_indices_bytes": kvi_h.numel() * 4,
        "h2d_indices_us": _median_wall(lambda: kvi_d.copy_(kvi_h, non_blocking=True), reps, torch),
        "h2d_q_bytes": q_h.numel() * 2,
        "h2d_q_us": _median_wall(lambda: q_d.copy_(q_h, non_blocking=True), reps, torch),
        "d2h_out_bytes": out_h.numel() * 2,
        "d2h_out_us": _median_wall(lambda: out_h.copy_(out_d, non_blocking=True), reps, torch),
        "empty_sync_us": _median_wall(lambda: None, reps, torch),
    }

    nbuf = binding.verify_attn_mla_host_buffer_size(case.qo_indptr, case.kv_indptr, H, 0)
    dbuf = torch.empty(nbuf, dtype=torch.uint8, device="cuda")
    host_call = binding.prepare_verify_attn_mla_host(q_h, dc.kv_pool, case.kv_indptr, kvi_h, case.qo_indptr,
                                                     out_h, lse_h, dbuf, case.sm_scale)
    for _ in range(3):
        host_call()
    res["host_call_us"] = _median_wall(host_call, reps, torch)

    out, lse = device.alloc_outputs(dc)
    ws = device.alloc_workspace(dc, 0)
    stream = torch.cuda.current_stream()
    call = binding.prepare_verify_attn_mla(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr,
                                           dc.kv_indptr_host, dc.qo_indptr_host, out, lse, ws, dc.sm_scale,
                                           stream=stream)
    for _ in range(3):
        call()
    res["device_call_us"] = _median_wall(call, reps, torch)

    host, dev = [], []
    for _ in range(reps):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200000)  # about 0.1 ms of GPU time: the call below queues behind it
        e0.record(stream)
        a = time.perf_counter()
        call()
        b = time.perf_counter()
        e1.record(stream)
        torch.cuda.synchronize()
        host.append((b - a) * 1e6)
        dev.append(e0.elapsed_time(e1) * 1e3)
    idle = []
    for _ in range(reps):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        idle.append(e0.elapsed_time(e1) * 1e3)
    res["submit"] = {"host_us": float(np.median(host)), "device_queued_us": float(np.median(dev)),
                     "from_idle_us": float(np.median(idle))}
    if binding.verify_attn_mla_check(ws) != 0:
        raise RuntimeError("kernel status")
    return res


def main(argv):
    names = argv or ["long_185k"]
    print(json.dumps([measure(n) for n in names], indent=1))


if __name__ == "__main__":
    main(sys.argv[1:])
