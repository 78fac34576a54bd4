"""Plain single-threaded CPU oracle for safetensors materialization.

Test infrastructure only (tests, smoke check, benchmark CPU baseline); the
product library never imports, links or calls it.
"""
