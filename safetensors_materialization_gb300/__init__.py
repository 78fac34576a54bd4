"""GB300-native safetensors materialization (``stmat``).

The C-ABI library ``libstmat.so`` (header parsing, views, planning, and the
sm_103a gather/cast kernels) is wrapped by :mod:`.stmat`; :mod:`.synth` builds
seeded synthetic checkpoints.
"""
