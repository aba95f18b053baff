"""Happens-before checker for the three-stream event protocol (test helper).

The hotdry.top page (section on the event-driven synchronisation protocol)
states what each event is for: Weights-Ready lets compute use a buffer only
after its weights arrived; Backward-Done lets the gradient stream export only
after the gradients exist; Buffer-Free lets the weight stream refill a buffer
only after its previous contents were consumed.  The same page and the
dimensionstp review (3-2 (4)) add pinned staging (packed by the host, read by
the copy) and the gradient slabs (written by the export, read by host Adam).

This checker replays an op list with vector clocks over the streams W, C, G,
the host thread H and the Adam dispatcher A, and asserts every data hazard
those sentences forbid is ordered:
  * H2D into buffer b after the previous compute on b and its export;
  * compute on b after this visit's H2D into b;
  * export from b after the compute that wrote its gradients;
  * host pack into staging b after the previous H2D read staging b;
  * D2H into slab k after the previous host job (Adam or FP32 accumulation)
    on slab k, the job after the D2H;
  * next step's pack / H2D of block j after block j's Adam;
  * MoE forward (lilting.ch, MoE section: only the routed experts are copied):
    the host reads the router's choice only after compute recorded it, the
    experts' copy into b follows every earlier use of b, and compute runs the
    experts only after that copy;
  * checkpoint slots: write after the previous save, save after the write;
    a host checkpoint is loaded only after it was saved and saved again only
    after its last load; a device checkpoint slot is refilled only after the
    last compute that read it, and read only after its load.
"""
from __future__ import annotations

STREAMS = ("W", "C", "G", "H", "A")


class Clock:
    def __init__(self, c=None):
        self.c = dict(c or {s: 0 for s in STREAMS})

    def merge(self, o: "Clock"):
        for k in self.c:
            self.c[k] = max(self.c[k], o.c[k])

    def copy(self):
        return Clock(self.c)


def _hb(a, b) -> bool:
    """True if op a (stream, clock) happens before op b."""
    if a is None:
        return True
    sa, ca = a
    _, cb = b
    return ca.c[sa] <= cb.c[sa]


def check(lines: list[str]) -> None:
    clk = {s: Clock() for s in STREAMS}
    ev: dict[str, Clock] = {}
    last_buf_use: dict[int, list] = {0: [], 1: []}     # ops that read/wrote device buffer b
    visit_h2d: dict[int, tuple] = {}                   # this visit's H2D into b
    exp_h2d: dict[int, tuple] = {}                     # this visit's routed-expert H2D into b
    route_rec: dict[int, tuple] = {}                   # compute's Route-Ready record of layer j
    slot_read: dict[int, tuple] = {}                   # compute that last read checkpoint slot q
    slot_load: dict[int, tuple] = {}                   # H2D_CKPT that last filled slot q
    slot_of_layer: dict[int, int] = {}                 # layer whose input X_{j-1} sits in slot q
    ckpt_saved: dict[int, tuple] = {}                  # D2H_CKPT of X_j into host memory
    ckpt_loaded: dict[int, tuple] = {}                 # H2D_CKPT that last read host X_j
    stage_read: dict[int, tuple] = {}                  # H2D that read staging b
    slab_adam: dict[int, tuple] = {}                   # Adam job that read slab k
    slab_d2h: dict[int, tuple] = {}
    adam_done: dict[int, tuple] = {}                   # block -> Adam job
    xslot_write: dict[int, tuple] = {}
    xslot_save: dict[int, tuple] = {}

    def tick(s):
        clk[s].c[s] += 1
        return (s, clk[s].copy())

    for ln, line in enumerate(lines):
        step, s, op, a, b = line.split()
        a, b = int(a), int(b)
        where = f"line {ln}: {line}"
        if s in ("W", "C", "G"):
            clk[s].merge(clk["H"])  # enqueued by the host after its earlier actions
        if op.startswith("WAIT_") and s in ("W", "C", "G"):
            name = op[5:] + str(a)
            if name in ev:
                clk[s].merge(ev[name])
            continue
        if op.startswith("REC_"):
            name = op[4:] + str(a)
            me = tick(s)
            ev[name] = me[1]
            if op == "REC_RT":
                route_rec[a] = me
            continue
        if s == "H":
            if op == "WAIT_ADAM":
                assert a in adam_done, where
                clk["H"].merge(adam_done[a][1])
            elif op == "WAIT_STAGE":
                # the staging buffer is free once every copy that read it is done:
                # the visit's H2D (Weights-Ready) and, for an MoE forward, the
                # routed experts' H2D (Experts-Ready)
                clk["H"].merge(ev["WR" + str(a)])
                if "ER" + str(a) in ev:
                    clk["H"].merge(ev["ER" + str(a)])
            elif op == "WAIT_RT":
                clk["H"].merge(ev["RT" + str(a)])
            elif op == "PACK_EXP":
                me = tick("H")
                assert _hb(route_rec.get(a), me) and a in route_rec, "experts packed before routing: " + where
            elif op == "PACK":
                me = tick("H")
                assert _hb(stage_read.get(b), me), "pack overwrites staging still being copied: " + where
                if a in adam_done:
                    assert _hb(adam_done[a], me), "pack before Adam of the block: " + where
            elif op == "ACQ_SLAB":
                if a in slab_adam:
                    clk["H"].merge(slab_adam[a][1])
            elif op in ("ADAM_ENQ", "ACCUM_ENQ"):
                # a host job on slab b: Adam (the step's last export of block a) or
                # the FP32 accumulation of an earlier micro-batch pass
                clk["A"].merge(clk["H"])
                clk["A"].merge(ev["SR" + str(b)])
                me = tick("A")
                assert _hb(slab_d2h[b], me), "host job reads slab before its D2H: " + where
                slab_adam[b] = me
                if op == "ADAM_ENQ":
                    adam_done[a] = me
            continue
        me = tick(s)
        if op == "H2D":
            for u in last_buf_use[b]:
                assert _hb(u, me), "H2D overwrites buffer still in use: " + where
            if a in adam_done:
                assert _hb(adam_done[a], me), "H2D of a block before its Adam: " + where
            visit_h2d[b] = me
            stage_read[b] = me
            last_buf_use[b] = [me]
        elif op == "H2D_EXP":
            assert a in route_rec and _hb(route_rec[a], me), "experts copied before the routing was read: " + where
            for u in last_buf_use[b]:
                assert _hb(u, me), "expert H2D overwrites buffer still in use: " + where
            if a in adam_done:
                assert _hb(adam_done[a], me), "expert H2D of a block before its Adam: " + where
            exp_h2d[b] = me
            stage_read[b] = me
            last_buf_use[b].append(me)
        elif op == "FWD_EXP":
            assert b in exp_h2d and _hb(exp_h2d[b], me), "experts computed before they arrived: " + where
            for u in last_buf_use[b]:
                assert _hb(u, me), "expert compute overlaps earlier use of buffer: " + where
            last_buf_use[b] = [me]
            del exp_h2d[b]
            xslot_write[a % 2] = me  # the combine writes X_j
        elif op == "H2D_CKPT":
            assert (a - 1) in ckpt_saved, "checkpoint loaded that was never saved: " + where
            assert _hb(ckpt_saved[a - 1], me), "checkpoint loaded before its save finished: " + where
            assert _hb(slot_read.get(b), me), "checkpoint H2D over a slot in use: " + where
            slot_load[b] = me
            slot_of_layer[a] = b
            ckpt_loaded[a - 1] = me
        elif op in ("FWD", "HEAD", "RECOMP", "BWD"):
            assert _hb(visit_h2d.get(b), me), "compute before weights ready: " + where
            for u in last_buf_use[b]:
                assert _hb(u, me), "compute overlaps earlier use of buffer: " + where
            last_buf_use[b] = [me]
            if op in ("RECOMP", "BWD") and a in slot_of_layer:
                q = slot_of_layer[a]
                assert _hb(slot_load[q], me), "compute reads a checkpoint slot before its load: " + where
                slot_read[q] = me
            if op == "FWD" or op == "HEAD":
                slot = a % 2
                if op == "FWD":
                    assert _hb(xslot_save.get(slot), me), "X slot overwritten before saved: " + where
                    xslot_write[slot] = me
        elif op == "D2H_CKPT":
            assert _hb(xslot_write[b], me), "checkpoint saved before written: " + where
            assert _hb(ckpt_loaded.get(a), me), "host checkpoint overwritten before its load: " + where
            xslot_save[b] = me
            ckpt_saved[a] = me
        elif op == "D2H":
            buf = _buf_of(lines, ln)
            assert _hb(last_buf_use[buf][-1], me), "export before gradients computed: " + where
            if b in slab_adam:
                assert _hb(slab_adam[b], me), "D2H into slab before its Adam finished: " + where
            slab_d2h[b] = me
            last_buf_use[buf].append(me)
        else:
            raise AssertionError("unknown op " + where)


def _buf_of(lines, ln):
    """Buffer of the export at line ln: the WAIT_BD just before it names it."""
    for k in range(ln - 1, -1, -1):
        p = lines[k].split()
        if p[1] == "G" and p[2] == "WAIT_BD":
            return int(p[3])
    raise AssertionError("export without Backward-Done wait")


def mask_slabs(lines: list[str]) -> list[str]:
    """The op list with slab numbers replaced by 'k'.  Which free slab an
    export takes is an allocation choice (it depends on when host Adam jobs
    finish); logs are compared modulo that choice and check() validates the
    actual assignment."""
    out = []
    for l in lines:
        step, s, op, a, b = l.split()
        if op in ("ACQ_SLAB", "REC_SR"):
            a = "k"
        elif op in ("D2H", "ADAM_ENQ", "ACCUM_ENQ"):
            b = "k"
        out.append(" ".join((step, s, op, a, b)))
    return out
