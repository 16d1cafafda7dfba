"""The device-side failure path of the tensor-core kernel, made to run on
purpose without faulting or hanging the GPU: ssd_fwd_fault_inject() stops the
kernel's TMA producer from issuing loads and caps every bounded wait at a
short count of polls.  The waits that depend on the loads run out,
the kernel records SSD_ERR_TIMEOUT with the code of the wait, every CTA drains
and frees its tensor memory and exits; the status is read and cleared on the
host, and the next ordinary call on the same workspace is correct."""
import pytest
import torch

import oracle
import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import synth

from gpu_helpers import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu
SSD_ERR_TIMEOUT = 5


@pytest.mark.parametrize("batch,seqlen,nheads,split_len,launches", [
    (1, 1024, 4, 1024, 1),    # one split: a single full-pass launch
    (1, 1024, 4, 256, 3),     # split plan: aggregate pass, composition, full pass
    (1, 512, 80, 128, 3),     # short splits on the persistent grid
])
def test_injected_stall_times_out_and_the_next_call_is_clean(batch, seqlen, nheads, split_len, launches):
    p = synth.make_problem(batch=batch, seqlen=seqlen, nheads=nheads, headdim=64, dstate=128, ngroups=1,
                           chunk=128, split_len=split_len, dtype="bf16", seed=21, init_std=0.1,
                           name=f"stall_b{batch}_L{seqlen}_H{nheads}_split{split_len}")
    d = to_device(p)
    f = ssd.SSDForward(p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, split_len, 0,
                       torch.bfloat16, "cuda")
    fam, n, _ = f.plan(True, True)
    assert fam == 1 and n == launches
    fin = torch.empty((p.batch, p.nheads, p.headdim, p.dstate), dtype=torch.float32, device="cuda")
    f.fault_inject(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], None, final_states=fin,
                   max_wait_rounds=1 << 14)
    st, where = f.check_status_where()
    # a wait code of the full-pass kernel (1-13) or of the split-aggregate kernel (21-25)
    assert st == SSD_ERR_TIMEOUT and (1 <= where <= 15 or 21 <= where <= 26), (st, where)
    assert f.check_status_where() == (0, 0)   # read once, then cleared
    # the GPU and the workspace serve the next ordinary call
    y = f(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], None, final_states=fin)
    assert f.check_status() == 0
    torch.cuda.synchronize()
    y_o, f_o = oracle.ssd_recurrence(p)
    ey = rel_err(y.float().cpu().numpy(), y_o)
    ef = rel_err(fin.cpu().numpy(), f_o)
    print(f"{p.name}: timeout at wait {where}; next call err_y={ey:.2e} err_state={ef:.2e}")
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"]
